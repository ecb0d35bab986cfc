// flush_wgen32.cu -- bucket-flush launchers and kernels of the generic row
// loop for bf16 terms at 32 ranks or more (rows loaded 8 at a time, batch 1),
// both output types.
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE_BF16_IN(dpred::kGenericLarge)
