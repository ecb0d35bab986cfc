// allgather.cu -- AllGather layouts (canonical and ring chunk order).
//
// Page "AllGather" (tier6-model interconnect notes): section "语义定义"
// (eq. ag-semantic-output, every node ends with [A_0, ..., A_{N-1}]) and
// section "Ring AllGather" (after the ring schedule node i holds
// [A_i, A_{i-1}, ..., A_{i-N+1}]).  On one GPU the N nodes are N output rows;
// each shard is read from HBM once and written N times, so the kernel moves
// M bytes in and N * M bytes out, the minimum for this layout.
#include "common.cuh"
#include "tma.cuh"

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
    int64_t items = (int64_t)n_nodes * shard_v;
    int64_t need = (items + kThreads - 1) / kThreads;
    int64_t g = (int64_t)sm_count() * resident_ctas(reinterpret_cast<const void*>(k), kThreads);
    if (need < g) g = need;
    if (g < 1) g = 1;
    k<<<(unsigned)g, kThreads, 0, s>>>(static_cast<const V*>(in), static_cast<V*>(out), n_nodes, shard_v, order);
    return DPRED_OK;
}

// TMA form: one thread per CTA moves 16 KB tiles.  Each tile of shard j is
// bulk-loaded once into a ring of shared-memory stages and bulk-stored from
// there to its N destinations (one bulk async-group per tile).  Loads run
// kLookahead tiles ahead of the stores; a stage is refilled only after the
// stores of the tile that last used it have finished reading it.
constexpr int kAgStages = 8;
constexpr int kAgLookahead = 4;
constexpr uint32_t kAgTile = 16384;

__global__ void __launch_bounds__(32, 1) allgather_tma_kernel(const char* __restrict__ in, char* __restrict__ out,
                                                               int n_nodes, int64_t shard_bytes, int order, int* err) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kAgStages];
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kAgStages; ++s) tma::mbar_init(&full[s], 1);
    tma::fence_barrier_init();
    const int64_t tiles_per_shard = (shard_bytes + kAgTile - 1) / kAgTile;
    const int64_t total = tiles_per_shard * n_nodes;
    const int64_t row = (int64_t)n_nodes * shard_bytes;
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
    const int64_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_of = [&](int64_t q, int& j, int64_t& off, uint32_t& bytes) {
        const int64_t t = blockIdx.x + q * gridDim.x;
        j = (int)(t / tiles_per_shard);
        off = (t - (int64_t)j * tiles_per_shard) * kAgTile;
        const int64_t rem = shard_bytes - off;
        bytes = (uint32_t)(rem < kAgTile ? rem : kAgTile);
    };
    auto issue_load = [&](int64_t q) {
        int j;
        int64_t off;
        uint32_t bytes;
        tile_of(q, j, off, bytes);
        const int s = (int)(q % kAgStages);
        tma::mbar_arrive_expect_tx(&full[s], bytes);
        tma::bulk_load(smem + (size_t)s * kAgTile, in + (int64_t)j * shard_bytes + off, bytes, &full[s]);
    };
    for (int64_t q = 0; q < mine && q < kAgLookahead; ++q) issue_load(q);
    for (int64_t q = 0; q < mine; ++q) {
        const int s = (int)(q % kAgStages);
        if (!tma::mbar_wait(&full[s], (uint32_t)((q / kAgStages) & 1))) {
            if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
            // let the loads already issued land (bounded) before leaving
            for (int64_t p = q + 1; p < mine && p < q + kAgLookahead; ++p)
                tma::mbar_wait(&full[p % kAgStages], (uint32_t)((p / kAgStages) & 1));
            break;
        }
        int j;
        int64_t off;
        uint32_t bytes;
        tile_of(q, j, off, bytes);
        for (int i = 0; i < n_nodes; ++i) {
            const int c = order == 0 ? j : (i - j + n_nodes) % n_nodes;
            tma::bulk_store(out + i * row + (int64_t)c * shard_bytes + off, smem + (size_t)s * kAgTile, bytes);
        }
        tma::bulk_commit();
        const int64_t nq = q + kAgLookahead;
        if (nq < mine) {
            // stage of tile nq was last used by tile nq - kAgStages: its stores must be done reading
            tma::bulk_wait_read<kAgStages - kAgLookahead - 1>();
            issue_load(nq);
        }
    }
    tma::bulk_wait<0>();  // every store complete before the CTA's shared memory goes away
}

}  // namespace

int launch_allgather(int n_nodes, int64_t shard_elems, int esize, const void* in, void* out, int order,
                     cudaStream_t s) {
    if (shard_elems == 0) return DPRED_OK;
    const int64_t shard_bytes = shard_elems * esize;
    const bool v16 = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0) &&
                     (shard_bytes % 16 == 0);
    if (v16 && flush_path() != PATH_LDG) {  // auto: the TMA form measured faster on GB300
        constexpr size_t smem = (size_t)kAgStages * kAgTile;
        static bool attr[64] = {};
        cudaError_t ea = ensure_smem_attr(allgather_tma_kernel, (int)smem, attr);
        if (ea != cudaSuccess) return cuda_error(ea, "allgather shared-memory attribute");
        const int64_t tiles = ((shard_bytes + kAgTile - 1) / kAgTile) * n_nodes;
        const int64_t g = tiles < sm_count() ? tiles : sm_count();
        allgather_tma_kernel<<<(unsigned)g, 32, smem, s>>>(static_cast<const char*>(in), static_cast<char*>(out),
                                                            n_nodes, shard_bytes, order, device_error_word());
    } else if (v16)
        launch_v<uint4>(n_nodes, shard_bytes / 16, in, out, order, s);
    else if (esize == 4)
        launch_v<uint32_t>(n_nodes, shard_elems, in, out, order, s);
    else
        launch_v<uint16_t>(n_nodes, shard_elems, in, out, order, s);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "allgather kernel launch");
}

}  // namespace dpred
