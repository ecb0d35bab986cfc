// common.cuh -- internal declarations shared by the libdpred translation units.
//
// Element rule of every reduction in this library (the pages' "same reduction,
// same operand order per element"): widen each term to fp32, optionally
// pre-divide it by the number of ranks, add the terms in rank order starting
// from the rank-0 term, round once to the output type.  Every fp32 operation
// is written with an explicit round-to-nearest intrinsic so that no compiler
// contraction (FMA) can change a bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "dpred.h"

namespace dpred {

// ------------------------------------------------------------------ errors --

int set_error(int code, const char* fmt, ...);
int cuda_error(cudaError_t e, const char* what);

// ----------------------------------------------------------- device info ---

int sm_count();  // SMs of the current device (cached per device)
// Resident CTAs per SM of `kernel` (any __global__ function) launched with
// `threads` threads and no dynamic shared memory, on the current device;
// queried once per (kernel, threads, device) and cached.  At least 1.
int resident_ctas(const void* kernel, int threads);

// Apply a kernel's dynamic shared-memory limit once per device; `done` is that
// kernel's per-device flag array (the attribute is per device context).
template <typename K>
cudaError_t ensure_smem_attr(K kernel, int bytes, bool (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

// ---------------------------------------------------------- element math ---

// Pre-division modes: none, multiply by the exact reciprocal of a power-of-two
// rank count (bit-identical to dividing), IEEE division by any rank count.
enum PreDiv : int { PDIV_NONE = 0, PDIV_POW2 = 1, PDIV_DIV = 2, PDIV_DIV_EXACT = 3 };
// PDIV_DIV_EXACT is a compile-time mode of the kernels only (plans carry
// PDIV_DIV): the division-free quotient without its per-term check, for rank
// counts where that quotient equals IEEE division on every input, subnormal
// quotients included.  Exhaustive checks on the host:
//  - bf16 terms (split reciprocal), all 65,536 bf16 values, every count from 3
//    to 64 that is not a power of two: exactly 3, 5, 15, 17 and 51;
//  - fp32 terms (Markstein's step), all 2^32 inputs: every odd count from 3 to
//    63.  At an even count a subnormal quotient can fall exactly on a rounding
//    midpoint, which the step can miss.
__host__ __device__ constexpr bool bf16_split_exact(int w) { return w == 3 || w == 5 || w == 15 || w == 17 || w == 51; }
__host__ __device__ constexpr bool f32_markstein_exact(int w) { return w >= 3 && w <= 63 && (w & 1) != 0; }
// The rank counts whose flush kernels use the unchecked quotient: every exact
// count but bf16 51, which stays on the chunk-8 loop (kGenericLarge) with its
// check.  The library's self-test checks this quotient at every count.
__host__ __device__ constexpr bool flush_prediv_unchecked(int w, bool bf16_in) {
    return bf16_in ? (bf16_split_exact(w) && w < 32) : f32_markstein_exact(w);
}

// Pre-division of one term in the scalar paths: IEEE division for a rank
// count that is not a power of two, an exact multiply for a power of two.
__device__ __forceinline__ float pre_divide(float x, int mode, float wf, float inv_w) {
    if (mode == PDIV_POW2) return __fmul_rn(x, inv_w);
    if (mode == PDIV_DIV || mode == PDIV_DIV_EXACT) return __fdiv_rn(x, wf);
    return x;
}

// Division-free pre-division for a rank count w that is not a power of two
// (the vector paths).  Both forms return x / w rounded to nearest even --
// bit for bit what IEEE division gives -- for every input except a few tiny
// ones whose quotient can be subnormal.  Each form flags those (the bf16 form
// with its own check, the fp32 form with prediv_tiny), and a vector holding a
// flagged term is reduced again with IEEE division.  The library's self-test
// checks both forms, checks included, against IEEE division on every input.
//
// bf16 terms (8 significant bits): 1/w = c_hi + c_lo with c_hi holding the
// leading 16 bits of 1/w and c_lo = RN(1/w - c_hi).  x * c_hi has at most 24
// significant bits, so it is exact, and RN(x * c_lo + x * c_hi) is one fused
// step whose operand is within about 2^-40 (relative) of x / w.  For w not a
// power of two the quotient of an 8-bit significand by w is never closer than
// about 2^-31 (relative) to a rounding midpoint, so that step rounds the same
// way as the exact quotient.
__device__ __forceinline__ float div_rank_count_bf16(float x, float c_hi, float c_lo) {
    return __fmaf_rn(x, c_lo, __fmul_rn(x, c_hi));
}

// The same quotient with its own check.  The fused step is evaluated a
// second time with subnormal operands and results flushed to zero.  For a bf16
// term the two differ exactly when x, the product x * c_hi or the quotient is
// subnormal, or x is NaN.  Where they agree, the quotient is a normal number
// (or zero, or infinite) computed from an exact product, and the rounding
// argument above holds.  Where they differ, `tiny` is set and the caller
// divides with IEEE division instead.  This check takes two instructions per
// term (one fused multiply-add, one compare), against three integer
// instructions for prediv_tiny.
__device__ __forceinline__ float div_rank_count_bf16_checked(float x, float c_hi, float c_lo, bool& tiny) {
    const float p = __fmul_rn(x, c_hi);
    const float t = __fmaf_rn(x, c_lo, p);
    float tf;
    asm("fma.rn.ftz.f32 %0, %1, %2, %3;" : "=f"(tf) : "f"(x), "f"(c_lo), "f"(p));
    tiny |= tf != t;
    return t;
}

// fp32 terms: Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; J.-M. Muller et al., "Handbook of Floating-Point
// Arithmetic", division with a fused multiply-add).  With y = RN(1/w),
// q = RN(x y) lies within one ulp of x/w, the residual r = x - q w is exact in
// one FMA, and RN(q + r y) is the correctly rounded quotient whenever it is a
// normal number.  A zero residual (q exact, including signed zeros) and a
// non-finite one (x infinite or NaN) keep q.
__device__ __forceinline__ float div_rank_count_f32(float x, float w, float inv_w) {
    const float q = __fmul_rn(x, inv_w);
    const float r = __fmaf_rn(-q, w, x);
    const float q1 = __fmaf_rn(r, inv_w, q);
    return (r == 0.0f || !isfinite(r)) ? q : q1;
}

// 0 < |x| < 2^-120: the inputs the fp32 division-free form leaves to IEEE division.
__device__ __forceinline__ bool prediv_tiny(float x) {
    return (__float_as_uint(x) & 0x7FFFFFFFu) - 1u < 0x037FFFFFu;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values to a bf16x2 word (round to nearest even); `lo` goes to the
// low half, i.e. the lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&v);
}

// ------------------------------------------------------------ flush plan ---

// One task of a flush as the kernel sees it (built on the host).
struct TaskDesc {
    int64_t src_off;     // element offset of the task in every row
    int64_t numel;       // elements (> 0)
    int64_t unit_begin;  // first work unit of the task (prefix over the plan)
    int32_t dst_begin;   // first destination pointer in the plan's pointer pool
    int16_t ndst;        // destinations to write (0..world)
    uint8_t vec;         // 0 scalar; 1 16-byte vectors, destinations co-aligned; 1+s realigned by s elements
    uint8_t head;        // scalar elements before the first 16-byte aligned vector
};
static_assert(sizeof(TaskDesc) == 32, "TaskDesc layout");

struct FlushHeader {
    const void* grads;
    int* err;            // device error word (bounded waits that give up record DPRED_E_TIMEOUT)
    int64_t ld;          // row stride in elements
    int64_t total_units;
    int32_t world;
    int32_t n_tasks;
    int32_t pdiv;        // PreDiv
    float wf, inv_w;     // world as float, its reciprocal (exact for powers of two)
    int32_t unit_vec;    // 16-byte vectors per work unit of the vector path
    float c_hi, c_lo;    // 1/world split for the bf16 division-free quotient (prediv_split)
};

// The split of 1/world used by div_rank_count_bf16: c_hi = the leading 16
// significant bits of 1/world, c_lo = RN(1/world - c_hi).
void prediv_split(int world, float* c_hi, float* c_lo);

constexpr int kInlineTasks = 128;
constexpr int kInlineDst = 512;

// Plan carried inside the launch (kernel parameter space, read through the
// constant cache): no device workspace and no host-to-device copy.
struct FlushArgsInline {
    FlushHeader h;
    TaskDesc tasks[kInlineTasks];
    void* dst[kInlineDst];
};

// Plan in caller-provided device workspace.
struct FlushArgsWs {
    FlushHeader h;
    const TaskDesc* tasks;
    void* const* dst;
};

constexpr int kFlushThreads = 256;
// Resident flush CTAs per SM: the persistent grid is capped at this many per
// SM, and the kernels of these world sizes are compiled to fit them.  Measured
// by interleaved A/B on GB300 with the grid capped at 2, 3 or 4 CTAs per SM:
// - W=8: 3 is 3-5% faster than 4 on ReduceScatter of 1 GiB rows and on single
//   buckets of 512 MB and more, within 0.5% on the 402.8M step, and 1.8%
//   slower on a step of 98 small buckets; 2 is slower everywhere.  W=4
//   follows W=8 (same loads in flight per thread: 4 rows x 2 vectors).
// - W=2 keeps only 2 x 2 loads in flight per thread and needs 4 CTAs: capped
//   at 3 it lost 7% on 1 GB buckets.
// W=16 and the generic world size keep what their registers allow (2).
__host__ __device__ constexpr int flush_ctas_per_sm(int w) { return w == 2 ? 4 : (w == 4 || w == 8) ? 3 : 16; }
// Launches that write at least half as many bytes as they read (an AllReduce
// delivered to every rank) run 2 CTAs per SM at W=4 and W=8: in place at W=8,
// 0.952 of peak against 0.915 at 3 CTAs, while the owner form (writes about a
// third of the reads) was 6% slower at 2.
inline int flush_ctas_per_sm(int w, bool write_heavy) {
    const int c = flush_ctas_per_sm(w);
    return (write_heavy && (w == 4 || w == 8)) ? 2 : c;
}
// The matching __launch_bounds__ minimum (0 = none).  Without a bound the
// W=8 kernel's register count moved between 56 and 89 with small source
// changes, i.e. between 4 and 2 resident CTAs; an explicit minimum of 1 also
// changes the allocation, so the other world sizes pass 0.
__host__ __device__ constexpr int flush_min_blocks(int w) { return (w == 2 || w == 4 || w == 8) ? flush_ctas_per_sm(w) : 2; }
constexpr int kUnitVec = 256;      // 16-byte vectors per thread-block pass of the vector path (4 KB per row)
constexpr int kUnitScalar = 2048;  // elements per work unit of the scalar path

struct FlushLaunch {
    FlushHeader h;
    int in_dt, out_dt;
    const TaskDesc* tasks;   // host plan
    void* const* dst;        // host pointer pool
    int n_dst;
    void* workspace;         // device, used when the plan does not fit inline
    size_t workspace_bytes;
    bool realign;            // some task takes the realigned vector path
    bool ldg_only;           // register streaming only: an operand lives in host memory
    bool pdl;                // may overlap the previous launch on the stream (disjoint buckets only)
    bool write_heavy;        // the launch writes at least half as many bytes as it reads
};

// World sizes with an unrolled flush kernel of their own (every size from 2
// to 16); larger ones take the generic row loop (template world size 0).
__host__ __device__ constexpr bool flush_specialised(int w) { return w >= 2 && w <= 16; }
// Vectors each thread keeps in flight per replica row, by template world size
// (0 = generic, rows in chunks of 4) and input type: sized so that a thread has
// about 8 to 21 16-byte loads outstanding.  Interleaved A/B at 256 MB per
// replica, fraction of the copy peak by batch:
//   W=3 bf16  3 / 4 / 6 = 0.807 / 0.850 / 0.816;  fp32 3 / 4 / 6 = 0.920 / 0.889 / 0.909
//   W=5 bf16  2 / 3 / 4 = 0.845 / 0.864 / 0.880;  fp32 = 0.924 / 0.946 / 0.970
//   W=6 bf16  2 / 3 = 0.874 / 0.899;  fp32 0.938 / 0.953
//   W=7 bf16  2 / 3 = 0.894 / 0.922;  fp32 0.933 / 0.960
//   W=9 / 10 / 11 batch 1 / 2: bf16 0.828 / 0.899, 0.838 / 0.908, 0.846 / 0.920;
//                              fp32 0.920 / 0.974, 0.914 / 0.977, 0.916 / 0.960
//   generic (then W=9) bf16 2 / 3 = 0.787 / 0.748 (3 spills);  fp32 0.838 / 0.885
// Re-run once the division path carried the lighter checks (two instructions
// per bf16 term, none at the exact counts), batch 1 / 2 at W = 12 / 13 / 14 / 15:
//   bf16 0.864 / 0.880 / 0.876 / 0.941 -> 0.929 / 0.917 / 0.933 / 0.998;
//   fp32 0.921 / 0.925 / 0.922 / 0.929 -> 0.975 / 0.986 / 0.981 / 0.997;
//   bf16 W=9 batch 2 / 3 = 0.912 / 0.932; W=10 / 11 batch 3 lost 0.4 / 0.2
//   points, W=7 batch 4 lost 1.4, W=6 batch 4 gained 1.0 but spilled (bf16 to
//   fp32), so those keep their batches.
//   generic loop, bf16 terms, rows in chunks of 4 with batch 2 against chunks
//   of 8 with batch 1 (kGenericLarge): W = 17 / 20 / 24 / 28 = 0.827 / 0.870 /
//   0.886 / 0.894 against 0.798 / 0.831 / 0.890 / 0.867; W = 32 / 40 / 48 / 64
//   = 0.856 / 0.726 / 0.787 / 0.786 against 1.004 / 0.919 / 0.927 / 0.922.
//   fp32 terms keep batch 3 and chunks of 4 (batch 2: W = 17-28 lost 4-7%).
__host__ __device__ constexpr int flush_batch_of(int w_t, bool bf16_in) {
    return w_t == 3 ? (bf16_in ? 4 : 3)
         : w_t == 5 ? 4
         : (w_t == 6 || w_t == 7) ? 3
         : w_t == 9 ? (bf16_in ? 3 : 2)
         : (w_t == 10 || w_t == 11) ? 2
         : (w_t >= 12 && w_t <= 15) ? 2
         : (w_t == 0 || w_t == -2) ? (bf16_in ? 2 : 3)
         : (w_t == 2 || w_t == 4) ? 2 : 1;
}
// Launch one CTA per work unit instead of a persistent grid (the block
// scheduler then balances the SMs; a persistent grid hands every CTA the same
// share up front).  Interleaved A/B at 256 MB per replica row, fraction of
// the copy peak, persistent -> one CTA per unit:
//   W = 16 bf16 / fp32: 1.030 -> 1.073, 1.033 -> 1.078;
//   generic loop (w_t = 0): fp32 W = 17 / 24 / 28 / 40 / 48 / 64 = 0.949 / 0.973 /
//   0.955 / 0.869 / 0.711 / 0.918 -> 0.969 / 1.011 / 1.012 / 1.010 / 1.010 / 1.017,
//   bf16 W = 17 / 20 / 24 = 0.826 / 0.867 / 0.877 -> 0.832 / 0.876 / 0.887;
//   chunk-8 loop, powers of two: W = 32 / 64 = 0.985 / 0.904 -> 0.996 / 1.024,
//   other sizes lost 1-4% (W = 36-56), as did W = 3-14 (2-8%) and W = 8 (18%,
//   its units carry a quarter of the bytes of a W = 16 unit).
__host__ __device__ constexpr bool flush_grid_per_unit(int w_t, bool pow2_prediv) {
    return w_t == 0 || w_t == -2 || w_t == 16 || (w_t == -1 && pow2_prediv);
}
// Template world size of the generic loop for bf16 terms at kGenericLargeFrom
// ranks or more: batch 1, rows loaded 8 at a time.
constexpr int kGenericLarge = -1;
constexpr int kGenericLargeFrom = 32;
// Template world size of the generic loop (as w_t = 0) for the counts above 16
// that divide without a check (flush_prediv_unchecked).
constexpr int kGenericExact = -2;
// The template world size of the kernels that flush `world` ranks.
__host__ __device__ constexpr int flush_kernel_world(int world, bool bf16_in) {
    return flush_specialised(world)                 ? world
         : flush_prediv_unchecked(world, bf16_in)   ? kGenericExact
         : (bf16_in && world >= kGenericLargeFrom)  ? kGenericLarge
                                                    : 0;
}
// A rank count that is not a power of two can reach the kernels of this
// template world size (the generic loops, or an unrolled size that is not a
// power of two), so they need the division path.
__host__ __device__ constexpr bool may_divide(int w_t) { return w_t <= 0 || (w_t & (w_t - 1)) != 0; }
inline int flush_batch(int world, bool bf16_in) { return flush_batch_of(flush_kernel_world(world, bf16_in), bf16_in); }

// Work units of a plan task; vec_elems = input elements per 16-byte vector,
// unit_vec = vectors per unit (kUnitVec x the batch).
inline int64_t flush_task_units(const TaskDesc& t, int vec_elems, int unit_vec) {
    if (t.vec) {
        int64_t nbody = (t.numel - t.head) / vec_elems;
        int64_t u = (nbody + unit_vec - 1) / unit_vec;
        return u > 0 ? u : 1;
    }
    return (t.numel + kUnitScalar - 1) / kUnitScalar;
}

// Host-side plan of one flush launch.
struct Dest {
    int64_t src_off, numel;
    std::vector<void*> ptrs;  // delivered, non-empty destinations (element 0 of the task)
};

struct BuiltPlan {
    FlushHeader h;
    int in_dt, out_dt;
    bool realign = false;
    bool ldg_only = false;  // gradients or destinations in pinned host memory
    bool write_heavy = false;  // destination bytes >= half the replica-row bytes read
    std::vector<TaskDesc> tasks;
    std::vector<void*> pool;
};

void build_plan(int world, int in_dt, const void* grads, int64_t ld, int out_dt, int pre_div,
                const std::vector<Dest>& tasks, BuiltPlan& out);
// pdl: launch with programmatic stream serialisation (the caller guarantees
// that this flush shares no byte with the previous launch on the stream).
int launch_plan(const BuiltPlan& p, void* workspace, size_t workspace_bytes, cudaStream_t s, bool pdl = false);

// Validation, plan and probe of one partitioned flush (each task cut at the
// partition boundaries of part_size elements; piece destinations inside the
// ranks' partition buffers part_dst[world]).
int partitioned_plan(int32_t world, int32_t in_dtype, int32_t out_dtype, const void* grads, int64_t ld,
                     const dpred_task* tasks, int32_t n_tasks, const int64_t* flat_offset, int32_t n_params,
                     int64_t part_size, void* const* part_dst, std::vector<Dest>& plan, dpred_probe* probe);

int launch_flush_bf16_in(const FlushLaunch& L, cudaStream_t s);
int launch_flush_f32_in(const FlushLaunch& L, cudaStream_t s);

int launch_accumulate(int world, int64_t n, float* acc, int g_dt, const void* g, int first, int finalize,
                      float scale, float* total, cudaStream_t s);

int launch_accumulator_save(int world, int64_t n, const float* acc, float* total, cudaStream_t s);
int launch_accumulator_restore(int world, int64_t n, float* acc, const float* total, cudaStream_t s);

int launch_allgather(int n_nodes, int64_t shard_elems, int esize, const void* in, void* out, int order,
                     cudaStream_t s);
// AllGather kernel form (see dpred_set_allgather_form); set_allgather_form
// returns the previous form, or -1 for an unknown one.
enum AllGatherForm : int { AG_AUTO = 0, AG_REGISTER = 1, AG_TMA1 = 2, AG_TMA4 = 3, AG_STAGED = 4, AG_SKEW = 5, AG_SKEW8K = 6 };
int allgather_form();
int set_allgather_form(int form);

// Plan-driven byte copy (the relayout pass): triples of {src byte offset, dst byte offset, bytes}.
int launch_copy_plan(const char* src, char* dst, const std::vector<int64_t>& triples, void* workspace,
                     size_t workspace_bytes, cudaStream_t s);
size_t relayout_workspace_bytes(int64_t n_pieces);

int* device_error_word();  // device address of the error word (current device)

// DPRED_OK when `s` is not being captured into a CUDA graph; otherwise
// DPRED_E_INVAL (what names the plan).  A plan uploaded from host memory must
// not be captured: the captured copy would read the host plan again at every
// replay, long after the call that owned it.
int refuse_capture_of_upload(cudaStream_t s, const char* what);

// Kernel family used by the bucket flush (and ReduceScatter): see dpred_set_flush_path.
enum FlushPath : int { PATH_AUTO = 0, PATH_LDG = 1, PATH_TMA = 2 };
int flush_path();

#ifdef __CUDACC__
__device__ __forceinline__ void record_device_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Checked builds (-DDPRED_CHECKED=1) test every global access of the flush
// kernels against the task it belongs to before making it.  A failed test
// records DPRED_E_BOUNDS in the device error word, and the access is skipped:
// a load reads zeros, a store does not happen.  In the default build every
// test is the constant true and compiles away.
#ifndef DPRED_CHECKED
#define DPRED_CHECKED 0
#endif
__device__ __forceinline__ bool access_ok(bool ok, int* err) {
#if DPRED_CHECKED
    if (!ok) {
        record_device_error(err, DPRED_E_BOUNDS);
        return false;
    }
#else
    (void)ok;
    (void)err;
#endif
    return true;
}
#endif

}  // namespace dpred
