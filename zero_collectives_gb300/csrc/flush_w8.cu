// flush_w8.cu -- bucket-flush launchers and kernels for world size 8, all four
// input/output type pairs (one translation unit per world size, built in parallel).
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE(8)
