// flush_wgen.cu -- bucket-flush launchers and kernels for the world sizes
// without a kernel of their own (the generic row loop), all four
// input/output type pairs (one translation unit per world size, built in
// parallel).
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE(0)
