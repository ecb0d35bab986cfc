// flush_w11.cu -- bucket-flush launchers and kernels for world size 11, all four
// input/output type pairs (one translation unit per world size, built in parallel).
#include "flush_kernels.cuh"

DPRED_FLUSH_INSTANTIATE(11)
