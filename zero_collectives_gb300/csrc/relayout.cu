// relayout.cu -- the bucket relayout pass: a plan-driven byte copy.
//
// DeepSpeed issue #8700, "Describe alternatives you've considered":
// ncclReduceScatter over a bucket needs the bucket laid out contiguously by
// destination rank, which DeepCompile's arrival-order buckets are not, so a
// relayout pass has to run first.  This kernel is that pass: every replica row
// of the arrival-order bucket is rewritten rank-major (the elements bound for
// rank 0 in flat order, then rank 1, ...).  It is a pure copy; the
// partitioned flush (dpred_flush_bucket_partitioned) does the same delivery in
// one fused pass without it.
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace dpred {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kUnitBytes = 16384;
constexpr int kInlinePieces = 640;

struct Piece {
    int64_t src;         // byte offset from the source base
    int64_t dst;         // byte offset from the destination base
    int64_t bytes;
    int64_t unit_begin;  // first copy unit of the piece
};

struct CopyHeader {
    const char* src;
    char* dst;
    int64_t total_units;
    int32_t n;
    int32_t vec;  // every piece 16-byte aligned on both sides with a 16-byte multiple size
};

struct CopyArgsInline {
    CopyHeader h;
    Piece p[kInlinePieces];
};

struct CopyArgsWs {
    CopyHeader h;
    const Piece* p;
};

__device__ __forceinline__ const Piece& piece(const CopyArgsInline& a, int i) { return a.p[i]; }
__device__ __forceinline__ const Piece& piece(const CopyArgsWs& a, int i) { return a.p[i]; }

template <typename Args>
__global__ void __launch_bounds__(kThreads) copy_kernel(const __grid_constant__ Args a) {
    const CopyHeader& h = a.h;
    for (int64_t u = blockIdx.x; u < h.total_units; u += gridDim.x) {
        int lo = 0, hi = h.n - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (piece(a, mid).unit_begin <= u)
                lo = mid;
            else
                hi = mid - 1;
        }
        const Piece P = piece(a, lo);
        const int64_t b0 = (u - P.unit_begin) * kUnitBytes;
        const int64_t b1 = b0 + kUnitBytes < P.bytes ? b0 + kUnitBytes : P.bytes;
        if (h.vec) {
            const uint4* s = reinterpret_cast<const uint4*>(h.src + P.src);
            uint4* d = reinterpret_cast<uint4*>(h.dst + P.dst);
            for (int64_t v = b0 / 16 + threadIdx.x; v < b1 / 16; v += kThreads) __stcs(d + v, __ldcs(s + v));
        } else {
            const uint16_t* s = reinterpret_cast<const uint16_t*>(h.src + P.src);
            uint16_t* d = reinterpret_cast<uint16_t*>(h.dst + P.dst);
            for (int64_t v = b0 / 2 + threadIdx.x; v < b1 / 2; v += kThreads) d[v] = s[v];
        }
    }
}

template <typename K>
unsigned grid_for(K kernel, int64_t units) {
    int64_t g = (int64_t)sm_count() * resident_ctas(reinterpret_cast<const void*>(kernel), kThreads);
    return (unsigned)(units < g ? units : g);
}

}  // namespace

size_t relayout_workspace_bytes(int64_t n_pieces) {
    return n_pieces <= kInlinePieces ? 0 : sizeof(Piece) * (size_t)n_pieces;
}

// pieces: {src byte offset, dst byte offset, bytes}; all byte counts even.
int launch_copy_plan(const char* src, char* dst, const std::vector<int64_t>& triples, void* workspace,
                     size_t workspace_bytes, cudaStream_t s) {
    std::vector<Piece> plan;
    int64_t units = 0;
    int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
    for (size_t i = 0; i + 2 < triples.size(); i += 3) {
        const int64_t so = triples[i], doff = triples[i + 1], b = triples[i + 2];
        if (b <= 0) continue;
        if (so % 16 || doff % 16 || b % 16) vec = 0;
        plan.push_back(Piece{so, doff, b, units});
        units += (b + kUnitBytes - 1) / kUnitBytes;
    }
    if (plan.empty()) return DPRED_OK;
    CopyHeader h{src, dst, units, (int32_t)plan.size(), vec};
    cudaError_t e;
    if ((int)plan.size() <= kInlinePieces) {
        CopyArgsInline a;
        a.h = h;
        std::copy(plan.begin(), plan.end(), a.p);
        auto k = copy_kernel<CopyArgsInline>;
        k<<<grid_for(k, units), kThreads, 0, s>>>(a);
        e = cudaGetLastError();
    } else {
        const size_t need = sizeof(Piece) * plan.size();
        if (!workspace || workspace_bytes < need)
            return set_error(DPRED_E_SIZE, "relayout plan of %zu pieces needs %zu bytes of workspace, got %zu",
                             plan.size(), need, workspace_bytes);
        if (reinterpret_cast<uintptr_t>(workspace) % 16) return set_error(DPRED_E_ALIGN, "workspace must be 16-byte aligned");
        const int rc = refuse_capture_of_upload(s, "a relayout plan");
        if (rc != DPRED_OK) return rc;
        e = cudaMemcpyAsync(workspace, plan.data(), need, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_error(e, "relayout plan copy");
        CopyArgsWs a;
        a.h = h;
        a.p = static_cast<const Piece*>(workspace);
        auto k = copy_kernel<CopyArgsWs>;
        k<<<grid_for(k, units), kThreads, 0, s>>>(a);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "relayout kernel launch");
}

}  // namespace dpred
