// flush_w9.cu -- bucket-flush launchers and kernels for world size 9, all four
// input/output type pairs (one translation unit per world size, built in parallel).
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE(9)
