// flush_dispatch.cu -- picks the flush launcher for a plan's world size and
// type pair.  The launchers are compiled in flush_w*.cu; here they are extern
// templates, so this unit compiles no kernel.
#include "flush_kernels.cuh"

DPRED_FLUSH_DECLARE(2)
DPRED_FLUSH_DECLARE(3)
DPRED_FLUSH_DECLARE(4)
DPRED_FLUSH_DECLARE(5)
DPRED_FLUSH_DECLARE(6)
DPRED_FLUSH_DECLARE(7)
DPRED_FLUSH_DECLARE(8)
DPRED_FLUSH_DECLARE(9)
DPRED_FLUSH_DECLARE(10)
DPRED_FLUSH_DECLARE(11)
DPRED_FLUSH_DECLARE(12)
DPRED_FLUSH_DECLARE(13)
DPRED_FLUSH_DECLARE(14)
DPRED_FLUSH_DECLARE(15)
DPRED_FLUSH_DECLARE(16)
DPRED_FLUSH_DECLARE(0)
DPRED_FLUSH_DECLARE_BF16_IN(dpred::kGenericLarge)
DPRED_FLUSH_DECLARE(dpred::kGenericExact)

namespace dpred {
namespace {

template <typename Tin, typename Tout>
int launch_flush_typed(const FlushLaunch& L, cudaStream_t s) {
    constexpr bool kBf16 = std::is_same<Tin, __nv_bfloat16>::value;
    switch (L.h.world) {
        case 2: return launch_flush_w<2, flush_batch_of(2, kBf16), Tin, Tout>(L, s);
        case 3: return launch_flush_w<3, flush_batch_of(3, kBf16), Tin, Tout>(L, s);
        case 4: return launch_flush_w<4, flush_batch_of(4, kBf16), Tin, Tout>(L, s);
        case 5: return launch_flush_w<5, flush_batch_of(5, kBf16), Tin, Tout>(L, s);
        case 6: return launch_flush_w<6, flush_batch_of(6, kBf16), Tin, Tout>(L, s);
        case 7: return launch_flush_w<7, flush_batch_of(7, kBf16), Tin, Tout>(L, s);
        case 8: return launch_flush_w<8, flush_batch_of(8, kBf16), Tin, Tout>(L, s);
        case 9: return launch_flush_w<9, flush_batch_of(9, kBf16), Tin, Tout>(L, s);
        case 10: return launch_flush_w<10, flush_batch_of(10, kBf16), Tin, Tout>(L, s);
        case 11: return launch_flush_w<11, flush_batch_of(11, kBf16), Tin, Tout>(L, s);
        case 12: return launch_flush_w<12, flush_batch_of(12, kBf16), Tin, Tout>(L, s);
        case 13: return launch_flush_w<13, flush_batch_of(13, kBf16), Tin, Tout>(L, s);
        case 14: return launch_flush_w<14, flush_batch_of(14, kBf16), Tin, Tout>(L, s);
        case 15: return launch_flush_w<15, flush_batch_of(15, kBf16), Tin, Tout>(L, s);
        case 16: return launch_flush_w<16, flush_batch_of(16, kBf16), Tin, Tout>(L, s);
        default: {
            const int wk = flush_kernel_world(L.h.world, kBf16);
            if (wk == kGenericExact)
                return launch_flush_w<kGenericExact, flush_batch_of(kGenericExact, kBf16), Tin, Tout>(L, s);
            if constexpr (kBf16) {
                if (wk == kGenericLarge)
                    return launch_flush_w<kGenericLarge, flush_batch_of(kGenericLarge, true), Tin, Tout>(L, s);
            }
            return launch_flush_w<0, flush_batch_of(0, kBf16), Tin, Tout>(L, s);
        }
    }
}

}  // namespace

int launch_flush_bf16_in(const FlushLaunch& L, cudaStream_t s) {
    if (L.out_dt == DPRED_BF16) return launch_flush_typed<__nv_bfloat16, __nv_bfloat16>(L, s);
    return launch_flush_typed<__nv_bfloat16, float>(L, s);
}

int launch_flush_f32_in(const FlushLaunch& L, cudaStream_t s) {
    if (L.out_dt == DPRED_F32) return launch_flush_typed<float, float>(L, s);
    return launch_flush_typed<float, __nv_bfloat16>(L, s);
}

}  // namespace dpred
