// allgather.cu -- AllGather layouts (canonical and ring chunk order).
//
// Page "AllGather" (tier6-model interconnect notes): section "语义定义"
// (eq. ag-semantic-output, every node ends with [A_0, ..., A_{N-1}]) and
// section "Ring AllGather" (after the ring schedule node i holds
// [A_i, A_{i-1}, ..., A_{i-N+1}]).  On one GPU the N nodes are N output rows;
// each shard is read from HBM once and written N times, so the kernel moves
// M bytes in and N * M bytes out, the minimum for this layout.
#include "common.cuh"

namespace dpred {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Flat index f = j * S + k over the input (shard j, position k).  Shard j
// lands at chunk c of row i, where c = j (canonical) or c = (i - j) mod N (ring).
template <typename V>
__global__ void __launch_bounds__(kThreads) allgather_kernel(const V* __restrict__ in, V* __restrict__ out, int n_nodes,
                                                             int64_t shard, int order) {
    const int64_t total = (int64_t)n_nodes * shard;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    const int64_t row = (int64_t)n_nodes * shard;
    for (int64_t f0 = tid; f0 < total; f0 += nthreads * kUnroll) {
        V q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            int64_t f = f0 + u * nthreads;
            if (f < total) q[u] = __ldcs(in + f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            int64_t f = f0 + u * nthreads;
            if (f < total) {
                const int j = (int)(f / shard);
                const int64_t k = f - (int64_t)j * shard;
                for (int i = 0; i < n_nodes; ++i) {
                    int c = order == 0 ? j : (i - j + n_nodes) % n_nodes;
                    __stcs(out + i * row + (int64_t)c * shard + k, q[u]);
                }
            }
        }
    }
}

template <typename V>
int launch_v(int n_nodes, int64_t shard_v, const void* in, void* out, int order, cudaStream_t s) {
    auto k = allgather_kernel<V>;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, 0) != cudaSuccess || occ < 1) occ = 1;
    int64_t items = (int64_t)n_nodes * shard_v;
    int64_t need = (items + kThreads - 1) / kThreads;
    int64_t g = (int64_t)sm_count() * occ;
    if (need < g) g = need;
    if (g < 1) g = 1;
    k<<<(unsigned)g, kThreads, 0, s>>>(static_cast<const V*>(in), static_cast<V*>(out), n_nodes, shard_v, order);
    return DPRED_OK;
}

}  // namespace

int launch_allgather(int n_nodes, int64_t shard_elems, int esize, const void* in, void* out, int order,
                     cudaStream_t s) {
    if (shard_elems == 0) return DPRED_OK;
    const int64_t shard_bytes = shard_elems * esize;
    const bool v16 = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0) &&
                     (shard_bytes % 16 == 0);
    if (v16)
        launch_v<uint4>(n_nodes, shard_bytes / 16, in, out, order, s);
    else if (esize == 4)
        launch_v<uint32_t>(n_nodes, shard_elems, in, out, order, s);
    else
        launch_v<uint16_t>(n_nodes, shard_elems, in, out, order, s);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "allgather kernel launch");
}

}  // namespace dpred
