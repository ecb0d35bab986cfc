// flush_wgenx.cu -- bucket-flush launchers and kernels of the generic row
// loop for the rank counts above 16 that divide without a per-term check
// (flush_prediv_unchecked: fp32 terms at odd counts, bf16 terms at 17), all
// four input/output type pairs.
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE(dpred::kGenericExact)
