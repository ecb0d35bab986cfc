// flush_f32.cu -- bucket-flush kernels for fp32 gradients (fp32 or bf16 destinations).
#include "flush_kernels.cuh"

namespace dpred {

int launch_flush_f32_in(const FlushLaunch& L, cudaStream_t s) {
    if (L.out_dt == DPRED_F32) return launch_flush_typed<float, float>(L, s);
    return launch_flush_typed<float, __nv_bfloat16>(L, s);
}

}  // namespace dpred
