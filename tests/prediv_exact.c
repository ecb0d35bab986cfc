/* Host check of the flush kernels' division-free bf16 quotient: for every rank
 * count W from 3 to 64 that is not a power of two, the split-reciprocal
 * quotient fma(x, c_lo, x * c_hi) (c_hi = the leading 16 significant bits of
 * 1/W, c_lo = RN(1/W - c_hi)) is compared with IEEE division x / W on all
 * 65,536 bf16 bit patterns (NaNs skipped).  Prints one line per W:
 *   W mismatches mismatches_with_|x|>=2^-120 checked_mismatches
 * where the last count applies the kernels' check: the same fused step with
 * subnormal operands and result flushed to zero (the GPU's fma.rn.ftz,
 * emulated here by flushing before and after), and IEEE division wherever the
 * two results differ.  Compiled without contraction or fast math: every
 * operation is one IEEE single-precision step with gradual underflow, as on
 * the GPU. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}
static uint32_t to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}
static float flush_subnormal(float v) { return fabsf(v) < 0x1p-126f ? copysignf(0.0f, v) : v; }

int main(void) {
    for (int w = 3; w <= 64; ++w) {
        if ((w & (w - 1)) == 0) continue;
        const double inv = 1.0 / (double)w;
        int e = 0;
        const double m = frexp(inv, &e);
        const double hi = ldexp(floor(ldexp(m, 16)), e - 16);
        const float c_hi = (float)hi, c_lo = (float)(inv - hi);
        long bad = 0, bad_large = 0, bad_checked = 0;
        for (uint32_t h = 0; h < 65536u; ++h) {
            const float x = from_bits(h << 16);
            if (isnan(x)) continue;
            const float want = x / (float)w;
            const float p = x * c_hi;
            const float got = fmaf(x, c_lo, p);
            if (to_bits(got) != to_bits(want)) {
                ++bad;
                if (fabsf(x) >= 0x1p-120f) ++bad_large;
            }
            const float twin = flush_subnormal(fmaf(flush_subnormal(x), flush_subnormal(c_lo), flush_subnormal(p)));
            const float checked = (twin != got) ? x / (float)w : got;
            if (to_bits(checked) != to_bits(want)) ++bad_checked;
        }
        printf("%d %ld %ld %ld\n", w, bad, bad_large, bad_checked);
    }
    return 0;
}
