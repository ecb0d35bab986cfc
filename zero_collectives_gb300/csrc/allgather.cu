// allgather.cu -- AllGather layouts (canonical and ring chunk order).
//
// Page "AllGather" (tier6-model interconnect notes): section "语义定义"
// (eq. ag-semantic-output, every node ends with [A_0, ..., A_{N-1}]) and
// section "Ring AllGather" (after the ring schedule node i holds
// [A_i, A_{i-1}, ..., A_{i-N+1}]).  On one GPU the N nodes are N output rows;
// each shard is read from HBM once and written N times, so the kernel moves
// M bytes in and N * M bytes out, the minimum for this layout ("理论下界":
// the cost is the N·M output).
//
// Three kernel forms move the same bytes:
//  - register streaming: every thread loads 16-byte vectors of one shard and
//    stores each to its N destinations;
//  - bulk copies (TMA): shard tiles are bulk-loaded into a ring of shared-
//    memory stages and bulk-stored from there to the N destinations, by one
//    or several issuing lanes per CTA, each with its own ring and bulk group;
//  - staged warp stores: one lane bulk-loads tiles into the ring, and eight
//    warps copy each staged tile to the N destinations with 16-byte
//    streaming stores from shared memory.
#include "common.cuh"
#include "tma.cuh"

namespace dpred {
namespace {

int g_allgather_form = AG_AUTO;

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Destination chunk of shard j in row i: c = j (canonical) or, in ring order
// (out[i][c] = in[(i - c) mod N]), c = (i - j) mod N.
__device__ __forceinline__ int ring_chunk(int i, int j, int n, int order) {
    if (order == 0) return j;
    const int c = i - j;
    return c < 0 ? c + n : c;
}

// Register streaming, shard-major: the grid strides over the vectors of one
// shard at a time (no division per vector), kUnroll vectors per thread in
// flight, each stored to its N destinations.
template <typename V>
__global__ void __launch_bounds__(kThreads) allgather_kernel(const V* __restrict__ in, V* __restrict__ out, int n_nodes,
                                                             int64_t shard, int order) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    const int64_t row = (int64_t)n_nodes * shard;
    for (int j = 0; j < n_nodes; ++j) {
        const V* src = in + (int64_t)j * shard;
        for (int64_t k0 = tid; k0 < shard; k0 += nthreads * kUnroll) {
            V q[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t k = k0 + u * nthreads;
                if (k < shard) q[u] = __ldcs(src + k);
            }
            for (int i = 0; i < n_nodes; ++i) {
                V* dst = out + i * row + (int64_t)ring_chunk(i, j, n_nodes, order) * shard;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t k = k0 + u * nthreads;
                    if (k < shard) __stcs(dst + k, q[u]);
                }
            }
        }
    }
}

template <typename V>
int launch_v(int n_nodes, int64_t shard_v, const void* in, void* out, int order, cudaStream_t s) {
    auto k = allgather_kernel<V>;
    int64_t need = (shard_v + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
    int64_t g = (int64_t)sm_count() * resident_ctas(reinterpret_cast<const void*>(k), kThreads);
    if (need < g) g = need;
    if (g < 1) g = 1;
    k<<<(unsigned)g, kThreads, 0, s>>>(static_cast<const V*>(in), static_cast<V*>(out), n_nodes, shard_v, order);
    return DPRED_OK;
}

// Tile q of an issuer that owns tiles g, g + G, g + 2G, ... of the n_nodes
// shards cut into tiles of TILE bytes (the last tile of a shard may be short).
struct AgTiles {
    int64_t tiles_per_shard, shard_bytes;
    __device__ void at(int64_t t, uint32_t tile, int& j, int64_t& off, uint32_t& bytes) const {
        j = (int)(t / tiles_per_shard);
        off = (t - (int64_t)j * tiles_per_shard) * tile;
        const int64_t rem = shard_bytes - off;
        bytes = (uint32_t)(rem < tile ? rem : tile);
    }
};

// Bulk-copy form.  Lane 0 of each of the CTA's ISSUERS warps is an
// independent issuer with its own STAGES-deep ring of TILE-byte stages and its
// own bulk async-group: it bulk-loads its tiles LOOK ahead of the stores, and
// refills a stage only after the stores of the tile that last used it have
// finished reading it.  With ISSUERS = 1 this is one issuing thread per CTA.
template <int ISSUERS, int STAGES, int LOOK, uint32_t TILE>
__global__ void __launch_bounds__(32 * ISSUERS, 1)
    allgather_tma_kernel(const char* __restrict__ in, char* __restrict__ out, int n_nodes, int64_t shard_bytes,
                         int order, int* err) {
    static_assert(LOOK >= 1 && LOOK < STAGES, "lookahead must leave a stage for the stores");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_all[ISSUERS * STAGES];
    if ((threadIdx.x & 31) != 0) return;
    const int w = threadIdx.x >> 5;
    unsigned char* ring = smem + (size_t)w * STAGES * TILE;
    uint64_t* full = full_all + w * STAGES;
    for (int s = 0; s < STAGES; ++s) tma::mbar_init(&full[s], 1);
    tma::fence_barrier_init();
    const AgTiles tl{(shard_bytes + TILE - 1) / TILE, shard_bytes};
    const int64_t total = tl.tiles_per_shard * n_nodes;
    const int64_t G = (int64_t)gridDim.x * ISSUERS;
    const int64_t g = (int64_t)w * gridDim.x + blockIdx.x;  // neighbouring CTAs take neighbouring tiles
    const int64_t mine = total > g ? (total - g + G - 1) / G : 0;
    const int64_t row = (int64_t)n_nodes * shard_bytes;
    auto issue_load = [&](int64_t q) {
        int j;
        int64_t off;
        uint32_t bytes;
        tl.at(g + q * G, TILE, j, off, bytes);
        const int s = (int)(q % STAGES);
        tma::mbar_arrive_expect_tx(&full[s], bytes);
        tma::bulk_load(ring + (size_t)s * TILE, in + (int64_t)j * shard_bytes + off, bytes, &full[s]);
    };
    for (int64_t q = 0; q < mine && q < LOOK; ++q) issue_load(q);
    for (int64_t q = 0; q < mine; ++q) {
        const int s = (int)(q % STAGES);
        if (!tma::mbar_wait(&full[s], (uint32_t)((q / STAGES) & 1))) {
            if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
            // every load issued so far (tiles q .. q + LOOK - 1, this one
            // included) must land before the shared memory goes away: wait
            // on each once more, bounded
            for (int64_t p = q; p < mine && p < q + LOOK; ++p)
                tma::mbar_wait(&full[p % STAGES], (uint32_t)((p / STAGES) & 1));
            break;
        }
        int j;
        int64_t off;
        uint32_t bytes;
        tl.at(g + q * G, TILE, j, off, bytes);
        for (int i = 0; i < n_nodes; ++i)
            tma::bulk_store(out + i * row + (int64_t)ring_chunk(i, j, n_nodes, order) * shard_bytes + off,
                            ring + (size_t)s * TILE, bytes);
        tma::bulk_commit();
        const int64_t nq = q + LOOK;
        if (nq < mine) {
            // the stage of tile nq was last used by tile nq - STAGES: its stores must be done reading
            tma::bulk_wait_read<STAGES - LOOK - 1>();
            issue_load(nq);
        }
    }
    tma::bulk_wait<0>();  // every store complete before the CTA's shared memory goes away
}

// Bulk-copy form with rows skewed in time.  In the plain bulk-copy form the N
// stores of one tile go to addresses a whole output row apart (a power of two
// for power-of-two sizes), so at any moment every SM writes N blocks that the
// HBM address map sends to the same channels.  Here the single issuing thread
// keeps the last D = min(N, DMAX) tiles staged and, in step q, stores tile
// q - (i mod D) to row i: concurrent stores to neighbouring rows are then a row
// minus a few tiles apart.  Every tile is still loaded once and stored N times.
// A tile's stage is refilled only after the step that made its last store
// (D - 1 steps after its first) has finished reading it.
template <int STAGES, int LOOK, uint32_t TILE, int DMAX>
__global__ void __launch_bounds__(32, 1)
    allgather_skew_kernel(const char* __restrict__ in, char* __restrict__ out, int n_nodes, int64_t shard_bytes,
                          int order, int* err) {
    static_assert(LOOK >= 1 && STAGES >= LOOK + DMAX, "the ring must hold the lookahead and the skew window");
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ int64_t t_off[STAGES];    // shard offset of the staged tile
    __shared__ int t_shard[STAGES];      // its shard
    __shared__ uint32_t t_bytes[STAGES]; // its length
    if (threadIdx.x != 0) return;
    for (int s = 0; s < STAGES; ++s) tma::mbar_init(&full[s], 1);
    tma::fence_barrier_init();
    const AgTiles tl{(shard_bytes + TILE - 1) / TILE, shard_bytes};
    const int64_t total = tl.tiles_per_shard * n_nodes;
    const int64_t G = gridDim.x, g = blockIdx.x;
    const int64_t mine = total > g ? (total - g + G - 1) / G : 0;
    const int64_t row = (int64_t)n_nodes * shard_bytes;
    const int D = n_nodes < DMAX ? n_nodes : DMAX;
    auto issue_load = [&](int64_t q) {
        const int s = (int)(q % STAGES);
        int j;
        int64_t off;
        uint32_t bytes;
        tl.at(g + q * G, TILE, j, off, bytes);
        t_off[s] = off;
        t_shard[s] = j;
        t_bytes[s] = bytes;
        tma::mbar_arrive_expect_tx(&full[s], bytes);
        tma::bulk_load(ring + (size_t)s * TILE, in + (int64_t)j * shard_bytes + off, bytes, &full[s]);
    };
    for (int64_t q = 0; q < mine && q < LOOK; ++q) issue_load(q);
    for (int64_t q = 0; q < mine + D - 1; ++q) {
        if (q < mine && !tma::mbar_wait(&full[q % STAGES], (uint32_t)((q / STAGES) & 1))) {
            if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
            // the loads of tiles q .. q + LOOK - 1 may still be landing: wait
            // on each once more (bounded), and on the stores already issued
            for (int64_t p = q; p < mine && p < q + LOOK; ++p)
                tma::mbar_wait(&full[p % STAGES], (uint32_t)((p / STAGES) & 1));
            break;
        }
        for (int i = 0; i < n_nodes; ++i) {
            const int64_t p = q - i % D;
            if (p < 0 || p >= mine) continue;
            const int s = (int)(p % STAGES);
            const int j = t_shard[s];
            tma::bulk_store(out + i * row + (int64_t)ring_chunk(i, j, n_nodes, order) * shard_bytes + t_off[s],
                            ring + (size_t)s * TILE, t_bytes[s]);
        }
        tma::bulk_commit();
        const int64_t nq = q + LOOK;
        if (nq < mine) {
            // stage of tile nq last held tile nq - STAGES, stored for the last
            // time in step nq - STAGES + D - 1: at most STAGES - LOOK - DMAX
            // later steps may still be reading
            tma::bulk_wait_read<STAGES - LOOK - DMAX>();
            issue_load(nq);
        }
    }
    tma::bulk_wait<0>();  // every store complete before the CTA's shared memory goes away
}

// Staged warp stores.  Warp 0 lane 0 bulk-loads this CTA's tiles into a
// STAGES-deep ring (`full` counts the bytes); warps 1..8 copy each staged tile
// to the N destinations with 16-byte streaming stores and release the stage
// on `empty` (one arrival per warp).
constexpr int kStoreWarps = 8;
template <int STAGES, uint32_t TILE>
__global__ void __launch_bounds__(32 * (kStoreWarps + 1), 1)
    allgather_staged_kernel(const char* __restrict__ in, char* __restrict__ out, int n_nodes, int64_t shard_bytes,
                            int order, int* err) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ __align__(8) uint64_t empty[STAGES];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tma::mbar_init(&full[s], 1);
            tma::mbar_init(&empty[s], kStoreWarps);
        }
        abort_flag = 0;
        tma::fence_barrier_init();
    }
    __syncthreads();
    const AgTiles tl{(shard_bytes + TILE - 1) / TILE, shard_bytes};
    const int64_t total = tl.tiles_per_shard * n_nodes;
    const int64_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t row = (int64_t)n_nodes * shard_bytes;
    volatile int* abort_v = &abort_flag;
    if (threadIdx.x < 32) {  // producer warp: lane 0 issues
        if (threadIdx.x != 0) return;
        int64_t issued = 0;
        for (int64_t q = 0; q < mine; ++q) {
            const int s = (int)(q % STAGES);
            if (*abort_v || !tma::mbar_wait(&empty[s], (uint32_t)(((q / STAGES) & 1) ^ 1))) {
                if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
                *abort_v = 1;
                break;
            }
            int j;
            int64_t off;
            uint32_t bytes;
            tl.at(blockIdx.x + q * gridDim.x, TILE, j, off, bytes);
            tma::mbar_arrive_expect_tx(&full[s], bytes);
            tma::bulk_load(smem + (size_t)s * TILE, in + (int64_t)j * shard_bytes + off, bytes, &full[s]);
            ++issued;
        }
        // leave only after every load issued has landed (bounded)
        const int64_t pend = issued < STAGES ? issued : STAGES;
        for (int64_t q = issued - pend; q < issued; ++q)
            if (!tma::mbar_wait(&full[q % STAGES], (uint32_t)((q / STAGES) & 1))) {
                if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
                break;
            }
        return;
    }
    const int ct = threadIdx.x - 32, lane = threadIdx.x & 31;
    for (int64_t q = 0; q < mine; ++q) {
        const int s = (int)(q % STAGES);
        if (*abort_v || !tma::mbar_wait(&full[s], (uint32_t)((q / STAGES) & 1))) {
            if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
            *abort_v = 1;
            return;
        }
        int j;
        int64_t off;
        uint32_t bytes;
        tl.at(blockIdx.x + q * gridDim.x, TILE, j, off, bytes);
        const uint4* src = reinterpret_cast<const uint4*>(smem + (size_t)s * TILE);
        const int nv = (int)(bytes / 16);
        for (int i = 0; i < n_nodes; ++i) {
            uint4* dst = reinterpret_cast<uint4*>(out + i * row + (int64_t)ring_chunk(i, j, n_nodes, order) * shard_bytes + off);
            for (int v = ct; v < nv; v += kStoreWarps * 32) __stcs(dst + v, src[v]);
        }
        __syncwarp();
        if (lane == 0) tma::mbar_arrive(&empty[s]);
    }
}

template <typename K>
cudaError_t launch_smem_kernel(K k, bool (&attr)[64], size_t smem, int64_t tiles, int threads, const void* in,
                               void* out, int n_nodes, int64_t shard_bytes, int order, cudaStream_t s) {
    cudaError_t ea = ensure_smem_attr(k, (int)smem, attr);
    if (ea != cudaSuccess) return ea;
    const int64_t g = tiles < sm_count() ? tiles : sm_count();
    k<<<(unsigned)g, threads, smem, s>>>(static_cast<const char*>(in), static_cast<char*>(out), n_nodes, shard_bytes,
                                         order, device_error_word());
    return cudaGetLastError();
}

}  // namespace

int allgather_form() { return g_allgather_form; }

int set_allgather_form(int form) {
    if (form < AG_AUTO || form > AG_SKEW8K) return -1;
    const int prev = g_allgather_form;
    g_allgather_form = form;
    return prev;
}

int launch_allgather(int n_nodes, int64_t shard_elems, int esize, const void* in, void* out, int order,
                     cudaStream_t s) {
    if (shard_elems == 0) return DPRED_OK;
    const int64_t shard_bytes = shard_elems * esize;
    const bool v16 = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0) &&
                     (shard_bytes % 16 == 0);
    int form = g_allgather_form;
    if (form == AG_AUTO) form = flush_path() == PATH_LDG ? AG_REGISTER : AG_SKEW;
    if (!v16) form = AG_REGISTER;
    cudaError_t e = cudaSuccess;
    if (form == AG_TMA1) {
        constexpr uint32_t tile = 16384;
        constexpr size_t smem = (size_t)8 * tile;
        static bool attr[64] = {};
        e = launch_smem_kernel(allgather_tma_kernel<1, 8, 4, tile>, attr, smem, (shard_bytes + tile - 1) / tile * n_nodes,
                               32, in, out, n_nodes, shard_bytes, order, s);
    } else if (form == AG_TMA4) {
        constexpr uint32_t tile = 8192;
        constexpr size_t smem = (size_t)4 * 6 * tile;
        static bool attr[64] = {};
        const int64_t tiles = (shard_bytes + tile - 1) / tile * n_nodes;
        e = launch_smem_kernel(allgather_tma_kernel<4, 6, 3, tile>, attr, smem, (tiles + 3) / 4, 128, in, out,
                               n_nodes, shard_bytes, order, s);
    } else if (form == AG_SKEW) {
        constexpr uint32_t tile = 16384;
        constexpr size_t smem = (size_t)12 * tile;
        static bool attr[64] = {};
        e = launch_smem_kernel(allgather_skew_kernel<12, 3, tile, 8>, attr, smem,
                               (shard_bytes + tile - 1) / tile * n_nodes, 32, in, out, n_nodes, shard_bytes, order, s);
    } else if (form == AG_SKEW8K) {
        constexpr uint32_t tile = 8192;
        constexpr size_t smem = (size_t)20 * tile;
        static bool attr[64] = {};
        e = launch_smem_kernel(allgather_skew_kernel<20, 6, tile, 8>, attr, smem,
                               (shard_bytes + tile - 1) / tile * n_nodes, 32, in, out, n_nodes, shard_bytes, order, s);
    } else if (form == AG_STAGED) {
        constexpr uint32_t tile = 16384;
        constexpr size_t smem = (size_t)8 * tile;
        static bool attr[64] = {};
        e = launch_smem_kernel(allgather_staged_kernel<8, tile>, attr, smem, (shard_bytes + tile - 1) / tile * n_nodes,
                               32 * (kStoreWarps + 1), in, out, n_nodes, shard_bytes, order, s);
    } else if (v16) {
        launch_v<uint4>(n_nodes, shard_bytes / 16, in, out, order, s);
    } else if (esize == 4) {
        launch_v<uint32_t>(n_nodes, shard_elems, in, out, order, s);
    } else {
        launch_v<uint16_t>(n_nodes, shard_elems, in, out, order, s);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "allgather kernel launch");
}

}  // namespace dpred
