// ceiling.cu -- write-only fills that measure the device's HBM write ceiling.
//
// Not part of the pages' method.  The AllGather ([AG] "理论下界": its cost
// is the N·M output) and the accumulator restore are dominated by stores, so
// their roofline is the rate at which HBM absorbs writes, not the copy rate.
// These kernels write a constant pattern and nothing else, so that rate can
// be measured on its own, independently of the kernels it bounds:
//   method 0: every thread of a persistent grid issues 16-byte streaming
//             stores (st.global.cs.v4);
//   method 1: the same with 32-byte stores (st.global.cs.v8);
//   method 2: one lane of each of four warps per CTA bulk-stores a 16 KB
//             shared-memory tile (cp.async.bulk) over consecutive tiles.
// A second kernel streams a given mix of reads and writes with no dependency
// between them: the ceiling for a kernel whose traffic has that mix (the
// AllGather reads M and writes N·M).
#include "common.cuh"
#include "tma.cuh"

namespace dpred {
namespace {

constexpr int kFillThreads = 512;
constexpr int kFillUnroll = 4;

__global__ void __launch_bounds__(kFillThreads) fill_v4_kernel(uint4* __restrict__ dst, int64_t n, uint32_t pat) {
    const int64_t stride = (int64_t)gridDim.x * kFillThreads;
    int64_t i = (int64_t)blockIdx.x * kFillThreads + threadIdx.x;
    for (; i + (kFillUnroll - 1) * stride < n; i += kFillUnroll * stride) {
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u)
            asm volatile("st.global.cs.v4.b32 [%0], {%1, %1, %1, %1};" ::"l"(dst + i + u * stride), "r"(pat)
                         : "memory");
    }
    for (; i < n; i += stride)
        asm volatile("st.global.cs.v4.b32 [%0], {%1, %1, %1, %1};" ::"l"(dst + i), "r"(pat) : "memory");
}

// n counts 32-byte vectors; dst is 32-byte aligned.
__global__ void __launch_bounds__(kFillThreads) fill_v8_kernel(char* __restrict__ dst, int64_t n, uint32_t pat) {
    const int64_t stride = (int64_t)gridDim.x * kFillThreads;
    int64_t i = (int64_t)blockIdx.x * kFillThreads + threadIdx.x;
    for (; i + (kFillUnroll - 1) * stride < n; i += kFillUnroll * stride) {
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u)
            asm volatile("st.global.cs.v8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"l"(dst + (i + u * stride) * 32),
                         "r"(pat)
                         : "memory");
    }
    for (; i < n; i += stride)
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"l"(dst + i * 32), "r"(pat)
                     : "memory");
}

constexpr uint32_t kFillTile = 16384;
constexpr int kFillIssuers = 4;

// bytes is a multiple of 16, dst 16-byte aligned.  Every issuer keeps at most
// 8 bulk groups outstanding.
__global__ void __launch_bounds__(32 * kFillIssuers, 1) fill_bulk_kernel(char* __restrict__ dst, int64_t bytes,
                                                                         uint32_t pat) {
    extern __shared__ __align__(128) unsigned char tile[];
    for (int i = threadIdx.x; i < (int)(kFillTile / 4); i += blockDim.x) reinterpret_cast<uint32_t*>(tile)[i] = pat;
    tma::fence_proxy_async_shared();  // the generic-proxy writes above, before the bulk stores read them
    __syncthreads();
    if ((threadIdx.x & 31) != 0) return;
    const int64_t tiles = (bytes + kFillTile - 1) / kFillTile;
    const int64_t G = (int64_t)gridDim.x * kFillIssuers;
    int n = 0;
    for (int64_t t = (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; t < tiles; t += G) {
        const int64_t off = t * kFillTile;
        const uint32_t b = (uint32_t)(bytes - off < kFillTile ? bytes - off : kFillTile);
        tma::bulk_store(dst + off, tile, b);
        tma::bulk_commit();
        if (++n >= 8) tma::bulk_wait_read<8>();
    }
    tma::bulk_wait<0>();
}

// Mixed streaming: write_bytes of a constant tile to dst and, spread evenly
// between those stores, read_bytes of src bulk-loaded into a ring of stages
// that nothing reads.  Loads and stores share no data, so no store waits for
// a load: the rate is what HBM sustains for this mix of reads and writes.
constexpr int kMixStages = 8;
__global__ void __launch_bounds__(32, 1) stream_mixed_kernel(const char* __restrict__ src, int64_t read_bytes,
                                                              char* __restrict__ dst, int64_t write_bytes, int* err) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ __align__(8) uint64_t full[kMixStages];
    unsigned char* tile = sm;              // the store tile
    unsigned char* ring = sm + kFillTile;  // load stages
    for (int i = threadIdx.x; i < (int)(kFillTile / 4); i += blockDim.x) reinterpret_cast<uint32_t*>(tile)[i] = 0x3F803F80u;
    tma::fence_proxy_async_shared();
    __syncwarp();
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kMixStages; ++s) tma::mbar_init(&full[s], 1);
    tma::fence_barrier_init();
    const int64_t G = gridDim.x, g = blockIdx.x;
    const int64_t wt = (write_bytes + kFillTile - 1) / kFillTile, rt = (read_bytes + kFillTile - 1) / kFillTile;
    const int64_t wmine = wt > g ? (wt - g + G - 1) / G : 0;
    const int64_t rmine = rt > g ? (rt - g + G - 1) / G : 0;
    const int64_t steps = wmine > rmine ? wmine : rmine;
    int64_t loads = 0;
    bool ok = true;
    for (int64_t q = 0; q < steps && ok; ++q) {
        // loads due by the end of step q: rmine * (q + 1) / steps
        const int64_t due = rmine * (q + 1) / steps;
        for (; loads < due; ++loads) {
            const int s = (int)(loads % kMixStages);
            if (loads >= kMixStages && !tma::mbar_wait(&full[s], (uint32_t)(((loads / kMixStages) - 1) & 1))) {
                ok = false;
                break;
            }
            const int64_t off = (g + loads * G) * kFillTile;
            const uint32_t b = (uint32_t)(read_bytes - off < kFillTile ? read_bytes - off : kFillTile);
            tma::mbar_arrive_expect_tx(&full[s], b);
            tma::bulk_load(ring + (size_t)s * kFillTile, src + off, b, &full[s]);
        }
        if (q < wmine) {
            const int64_t off = (g + q * G) * kFillTile;
            const uint32_t b = (uint32_t)(write_bytes - off < kFillTile ? write_bytes - off : kFillTile);
            tma::bulk_store(dst + off, tile, b);
            tma::bulk_commit();
            tma::bulk_wait_read<8>();
        }
    }
    if (!ok && err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
    // every load issued lands before the shared memory goes away (bounded)
    for (int64_t p = loads > kMixStages ? loads - kMixStages : 0; p < loads; ++p)
        if (!tma::mbar_wait(&full[p % kMixStages], (uint32_t)((p / kMixStages) & 1))) {
            if (err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
            break;
        }
    tma::bulk_wait<0>();
}

}  // namespace
}  // namespace dpred

using namespace dpred;

extern "C" int dpred_stream_mixed(const void* src, size_t read_bytes, void* dst, size_t write_bytes, void* stream) {
    if (read_bytes + write_bytes == 0) return DPRED_OK;
    if ((read_bytes && !src) || (write_bytes && !dst)) return set_error(DPRED_E_INVAL, "null pointer");
    if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16 || read_bytes % 16 ||
        write_bytes % 16)
        return set_error(DPRED_E_ALIGN, "mixed stream needs 16-byte aligned buffers and sizes");
    static bool attr[64] = {};
    const int smem = (int)((1 + kMixStages) * kFillTile);
    cudaError_t e = ensure_smem_attr(stream_mixed_kernel, smem, attr);
    if (e == cudaSuccess) {
        const int64_t tiles = (int64_t)((read_bytes > write_bytes ? read_bytes : write_bytes) + kFillTile - 1) / kFillTile;
        const int64_t g = tiles < sm_count() ? tiles : sm_count();
        stream_mixed_kernel<<<(unsigned)g, 32, smem, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const char*>(src), (int64_t)read_bytes, static_cast<char*>(dst), (int64_t)write_bytes,
            device_error_word());
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "mixed stream kernel launch");
}

extern "C" int dpred_fill_pattern(void* dst, size_t bytes, uint32_t pattern, int32_t method, int32_t ctas_per_sm,
                                  void* stream) {
    if (method < 0 || method > 2) return set_error(DPRED_E_INVAL, "fill method %d: 0, 1 or 2", method);
    if (bytes == 0) return DPRED_OK;
    if (!dst) return set_error(DPRED_E_INVAL, "null destination");
    const size_t gran = method == 1 ? 32 : 16;
    if (reinterpret_cast<uintptr_t>(dst) % gran != 0 || bytes % gran != 0)
        return set_error(DPRED_E_ALIGN, "fill method %d needs a %zu-byte aligned destination and size", method, gran);
    if (ctas_per_sm < 0 || ctas_per_sm > 32) return set_error(DPRED_E_INVAL, "ctas_per_sm %d outside 0..32", ctas_per_sm);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (method == 2) {
        static bool attr[64] = {};
        e = ensure_smem_attr(fill_bulk_kernel, (int)kFillTile, attr);
        if (e == cudaSuccess) {
            const int64_t tiles = ((int64_t)bytes + kFillTile - 1) / kFillTile;
            int64_t g = (int64_t)sm_count() * (ctas_per_sm > 0 ? ctas_per_sm : 1);
            const int64_t need = (tiles + kFillIssuers - 1) / kFillIssuers;
            if (need < g) g = need;
            fill_bulk_kernel<<<(unsigned)g, 32 * kFillIssuers, kFillTile, s>>>(static_cast<char*>(dst), (int64_t)bytes,
                                                                                pattern);
        }
    } else {
        const void* k = method == 0 ? reinterpret_cast<const void*>(fill_v4_kernel)
                                    : reinterpret_cast<const void*>(fill_v8_kernel);
        const int occ = ctas_per_sm > 0 ? ctas_per_sm : resident_ctas(k, kFillThreads);
        const int64_t n = (int64_t)(bytes / gran);
        int64_t g = (int64_t)sm_count() * occ;
        const int64_t need = (n + kFillThreads - 1) / kFillThreads;
        if (need < g) g = need;
        if (method == 0)
            fill_v4_kernel<<<(unsigned)g, kFillThreads, 0, s>>>(static_cast<uint4*>(dst), n, pattern);
        else
            fill_v8_kernel<<<(unsigned)g, kFillThreads, 0, s>>>(static_cast<char*>(dst), n, pattern);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "fill kernel launch");
}
