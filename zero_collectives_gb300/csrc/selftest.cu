// selftest.cu -- exercises the device error paths without any fault.
//  * Bounded wait: one thread waits on an mbarrier phase that nothing will
//    complete, gives up after the given clock budget and records
//    DPRED_E_TIMEOUT in the device error word, exactly as a real flush wait
//    would.
//  * Bounds test: one thread runs the flush kernels' access test on an index
//    outside its range.  The checked build records DPRED_E_BOUNDS; the default
//    build compiles the test away.  Nothing is accessed in either build.
//  * Pre-division test: the flush's pre-division by a rank count (the
//    division-free quotients for counts that are not powers of two) against
//    IEEE division, on every fp32 bit pattern and every bf16 value.
#include "common.cuh"
#include "tma.cuh"

namespace {

__global__ void wait_timeout_kernel(int* err, long long budget) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        dpred::tma::mbar_init(&bar, 1);  // expects one arrival that never comes
        dpred::tma::fence_barrier_init();
        if (!dpred::tma::mbar_wait(&bar, 0, budget) && err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
    }
}

__global__ void bounds_test_kernel(int* err, int64_t n, int64_t idx) {
    (void)dpred::access_ok(idx >= 0 && idx < n, err);
}

__device__ unsigned long long g_prediv_mismatches;
__device__ unsigned int g_prediv_first;  // lowest mismatching bit pattern seen (0xFFFFFFFF: none)

// The quotient the flush kernels' vector paths use for one term: an exact
// multiply for a power-of-two rank count; otherwise the division-free form of
// the input type, or IEEE division for a tiny term.
__device__ float vector_prediv(float x, int mode, float w, float inv_w, float c_hi, float c_lo, bool bf16) {
    if (mode == dpred::PDIV_POW2) return __fmul_rn(x, inv_w);
    if (mode == dpred::PDIV_NONE) return x;
    if (dpred::flush_prediv_unchecked((int)w, bf16))
        return bf16 ? dpred::div_rank_count_bf16(x, c_hi, c_lo) : dpred::div_rank_count_f32(x, w, inv_w);
    if (bf16) {
        bool tiny = false;
        const float t = dpred::div_rank_count_bf16_checked(x, c_hi, c_lo, tiny);
        return tiny ? __fdiv_rn(x, w) : t;
    }
    if (dpred::prediv_tiny(x)) return __fdiv_rn(x, w);
    return dpred::div_rank_count_f32(x, w, inv_w);
}

// Inputs [base, base + gridDim.x * blockDim.x * per): bit pattern u -> float;
// every pattern is checked as an fp32 term, and the patterns whose low 16 bits
// are zero (the bf16 values) also as bf16 terms.
__global__ void prediv_test_kernel(float w, float inv_w, float c_hi, float c_lo, int mode, uint64_t base, int per) {
    unsigned long long bad = 0;
    const uint64_t t = base + ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * (uint64_t)per;
    for (int i = 0; i < per; ++i) {
        const uint32_t u = (uint32_t)(t + (uint64_t)i);
        const float x = __uint_as_float(u);
        const float want = mode == dpred::PDIV_NONE ? x : __fdiv_rn(x, w);
        for (int k = 0; k < ((u & 0xFFFFu) == 0 ? 2 : 1); ++k) {
            const float got = vector_prediv(x, mode, w, inv_w, c_hi, c_lo, k == 1);
            const bool same = __float_as_uint(got) == __float_as_uint(want) || (isnan(got) && isnan(want));
            if (!same) {
                ++bad;
                atomicMin(&g_prediv_first, u);
            }
        }
    }
    if (bad) atomicAdd(&g_prediv_mismatches, bad);
}

}  // namespace

extern "C" int dpred_selftest_prediv(int32_t world, uint64_t* mismatches, uint32_t* first_mismatch) {
    if (world < 1 || world > DPRED_MAX_WORLD) return dpred::set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (!mismatches || !first_mismatch) return dpred::set_error(DPRED_E_INVAL, "null output");
    const unsigned long long zero = 0;
    const unsigned int none = 0xFFFFFFFFu;
    cudaError_t e = cudaMemcpyToSymbol(g_prediv_mismatches, &zero, sizeof zero);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_prediv_first, &none, sizeof none);
    const int mode = world == 1 ? dpred::PDIV_NONE : ((world & (world - 1)) == 0 ? dpred::PDIV_POW2 : dpred::PDIV_DIV);
    const float w = (float)world, inv_w = 1.0f / (float)world;
    float c_hi = 0.0f, c_lo = 0.0f;
    dpred::prediv_split(world, &c_hi, &c_lo);
    // 2^32 inputs: 2^14 blocks x 256 threads x 1024 inputs each
    constexpr int kBlocks = 1 << 14, kThreads = 256, kPer = 1024;
    if (e == cudaSuccess) {
        prediv_test_kernel<<<kBlocks, kThreads>>>(w, inv_w, c_hi, c_lo, mode, 0, kPer);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    unsigned long long n = 0;
    unsigned int f = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&n, g_prediv_mismatches, sizeof n);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&f, g_prediv_first, sizeof f);
    if (e != cudaSuccess) return dpred::cuda_error(e, "pre-division self-test");
    *mismatches = n;
    *first_mismatch = f;
    return DPRED_OK;
}

extern "C" int dpred_selftest_bounds(void* stream) {
    int* err = dpred::device_error_word();
    if (!err) return dpred::set_error(DPRED_E_CUDA, "device error word unavailable");
    bounds_test_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err, 16, 16);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "self-test launch");
}

extern "C" int dpred_selftest_wait_timeout(int64_t budget_cycles, void* stream) {
    if (budget_cycles < 0 || budget_cycles > 4000000000LL)
        return dpred::set_error(DPRED_E_INVAL, "budget %lld cycles outside 0..4e9", (long long)budget_cycles);
    int* err = dpred::device_error_word();
    if (!err) return dpred::set_error(DPRED_E_CUDA, "device error word unavailable");
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, budget_cycles);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "self-test launch");
}
