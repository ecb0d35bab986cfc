// flush_bf16.cu -- bucket-flush kernels for bf16 gradients (bf16 or fp32 destinations).
#include "flush_kernels.cuh"

namespace dpred {

int launch_flush_bf16_in(const FlushLaunch& L, cudaStream_t s) {
    if (L.out_dt == DPRED_BF16) return launch_flush_typed<__nv_bfloat16, __nv_bfloat16>(L, s);
    return launch_flush_typed<__nv_bfloat16, float>(L, s);
}

}  // namespace dpred
