// flush_kernels.cuh -- the bucket-flush kernel (reduce to owner / AllReduce
// fallback / empty-buffer skip), shared by ReduceScatter.
//
// DeepSpeed issue #8700 "[REQUEST] DeepCompile ZeRO-1: reduce-to-owner instead
// of AllReduce": each bucket task is one whole parameter; its reduced value
// goes to the owner's buffer only (ncclReduce(root=owner)) or, for a parameter
// straddling a partition boundary, to every rank's buffer (ncclAllReduce), and
// empty buffers are skipped in the copy-out.  On one GPU the W replicas are W
// rows of the bucket, so the "collective" is a streaming reduction over the
// rows whose store goes straight into the delivered, non-empty destinations:
// the copy-out is fused into the store.
//
// Work decomposition: the host cuts every task into work units (256 16-byte
// vectors on the vector path, 2048 elements on the scalar path); a persistent
// grid strides over units in bucket order and finds each unit's task by a
// binary search over the plan (all threads of a CTA read the same entries, a
// broadcast from the constant cache).  Each thread keeps W x BATCH 16-byte
// loads in flight, then reduces them in rank order.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "tma.cuh"

namespace dpred {

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;  // elements per 16-byte vector
    __device__ static float load(const __nv_bfloat16* p) {
        return bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(p));
    }
    __device__ static void store(__nv_bfloat16* p, float v) { *reinterpret_cast<uint16_t*>(p) = f32_to_bf16_bits(v); }
};
template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    __device__ static float load(const float* p) { return *p; }
    __device__ static void store(float* p, float v) { *p = v; }
};

template <typename Args>
__device__ __forceinline__ int64_t h_unit(const Args& a) { return a.h.unit_vec; }

__device__ __forceinline__ const TaskDesc& plan_task(const FlushArgsInline& a, int i) { return a.tasks[i]; }
__device__ __forceinline__ const TaskDesc& plan_task(const FlushArgsWs& a, int i) { return a.tasks[i]; }
__device__ __forceinline__ void* plan_dst(const FlushArgsInline& a, int i) { return a.dst[i]; }
__device__ __forceinline__ void* plan_dst(const FlushArgsWs& a, int i) { return a.dst[i]; }

// Unpack one 16-byte input vector into fp32 values.
template <typename Tin>
__device__ __forceinline__ void unpack(const uint4& q, float (&f)[Elem<Tin>::kVec]);
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4& q, float (&f)[8]) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x);
    f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z);
    f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
}
template <>
__device__ __forceinline__ void unpack<float>(const uint4& q, float (&f)[4]) {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
}

// Store VEC reduced values (already rounded in the caller's order) to dst.
template <typename Tout, int VEC>
__device__ __forceinline__ void store_vec(Tout* p, const float (&y)[VEC]);
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16, 8>(__nv_bfloat16* p, const float (&y)[8]) {
    uint4 q = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                         pack_bf16x2(y[6], y[7]));
    __stcs(reinterpret_cast<uint4*>(p), q);
}
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16, 4>(__nv_bfloat16* p, const float (&y)[4]) {
    uint2 q = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
    __stcs(reinterpret_cast<uint2*>(p), q);
}
template <>
__device__ __forceinline__ void store_vec<float, 8>(float* p, const float (&y)[8]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(y[0], y[1], y[2], y[3]));
    __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(y[4], y[5], y[6], y[7]));
}
template <>
__device__ __forceinline__ void store_vec<float, 4>(float* p, const float (&y)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(y[0], y[1], y[2], y[3]));
}

// A 16-byte load of a replica row that a checked build skips (reads zeros)
// when its bounds test failed; see access_ok.  Rows are loaded cached in L2
// at normal priority (ld.global.cg); results are stored evict-first
// (st.global.cs).  Interleaved A/B on GB300 at the same occupancy (3 CTAs per
// SM, W=8) against evict-first (.cs) loads: 3.7% faster on 64 MB-per-replica
// buckets, within 0.5% on the 402.8M step, ReduceScatter and 1 GB buckets,
// 1.4% slower on a step of 98 small buckets.  Non-coherent loads and L2
// 256-byte prefetch hints were no better; plain and .cg stores were 3-7%
// slower than .cs stores.
__device__ __forceinline__ uint4 load_vec(const uint4* p, bool ok) {
#if DPRED_CHECKED
    return ok ? __ldcg(p) : make_uint4(0u, 0u, 0u, 0u);
#else
    return __ldcg(p);
#endif
}

// The kernels' mode for a plan that divides: none where the template world
// size never divides, the unchecked quotient at the counts that take it
// (flush_prediv_unchecked, and the kGenericExact loop), else the checked one.
template <typename Tin>
__host__ __device__ constexpr int div_mode(int w_t) {
    return !may_divide(w_t) ? PDIV_NONE
         : (w_t == kGenericExact || (w_t > 0 && flush_prediv_unchecked(w_t, std::is_same<Tin, __nv_bfloat16>::value)))
             ? PDIV_DIV_EXACT
             : PDIV_DIV;
}

// Fold one replica's vector into the running sums (rank order is the call
// order).  With a rank count that is not a power of two the terms take the
// division-free quotient, and `tiny` is set when one of them needs IEEE
// division instead (see prediv_tiny); the caller then reduces the vector
// again with reduce_vec_ieee.
template <typename Tin, int MODE>
__device__ __forceinline__ void fold(float (&y)[Elem<Tin>::kVec], const uint4& q, bool first, const FlushHeader& h,
                                     bool& tiny) {
    constexpr int VEC = Elem<Tin>::kVec;
    constexpr bool kBf16 = std::is_same<Tin, __nv_bfloat16>::value;
    float f[VEC];
    unpack<Tin>(q, f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        if constexpr (kBf16 && MODE == PDIV_POW2) {
            // x * 2^-k is exact for a bf16 x (8 significant bits, lowest bit at
            // 2^-133 or above; 2^-133 * 2^-6 is still a multiple of the smallest
            // fp32 subnormal 2^-149) and 2^k <= 64 ranks.  So rounding
            // x * inv_w + y once gives the bits of rounding y + (x / W): one
            // fused step instead of a multiply and an add.  fp32 inputs keep
            // the two steps, since their quotient can be inexact.
            y[j] = first ? __fmul_rn(f[j], h.inv_w) : __fmaf_rn(f[j], h.inv_w, y[j]);
        } else if constexpr (MODE == PDIV_DIV_EXACT) {
            const float t = kBf16 ? div_rank_count_bf16(f[j], h.c_hi, h.c_lo) : div_rank_count_f32(f[j], h.wf, h.inv_w);
            y[j] = first ? t : __fadd_rn(y[j], t);
        } else if constexpr (MODE == PDIV_DIV) {
            float t;
            if constexpr (kBf16) {
                t = div_rank_count_bf16_checked(f[j], h.c_hi, h.c_lo, tiny);
            } else {
                t = div_rank_count_f32(f[j], h.wf, h.inv_w);
                tiny |= prediv_tiny(f[j]);
            }
            y[j] = first ? t : __fadd_rn(y[j], t);
        } else {
            const float t = pre_divide(f[j], MODE, h.wf, h.inv_w);
            y[j] = first ? t : __fadd_rn(y[j], t);
        }
    }
}

// The rows of one vector reduced again term by term with IEEE division, for
// the rare vector that holds a tiny term (rows in global memory, or staged in
// shared memory row_bytes apart).  The global-memory form is a function of its
// own, called only for such a vector and returning its values by value: kept
// out of the unrolled row loops, it shortened the hot code (interleaved A/B
// at 256 MB per replica, inline -> out of line: bf16 W=3 0.850 -> 0.861,
// W=13 0.831 -> 0.881, fp32 W=6 0.954 -> 0.973; W=12 unchanged).
template <int VEC>
struct VecF {
    float v[VEC];
};

template <typename Tin>
__device__ __noinline__ VecF<Elem<Tin>::kVec> reduce_vec_ieee_out(const uint4* base, int64_t stride, int64_t v,
                                                                  int world, float wf, bool ok) {
    constexpr int VEC = Elem<Tin>::kVec;
    VecF<VEC> y;
#pragma unroll 1
    for (int r = 0; r < world; ++r) {
        float f[VEC];
        unpack<Tin>(load_vec(base + (int64_t)r * stride + v, ok), f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float t = __fdiv_rn(f[j], wf);
            y.v[j] = r == 0 ? t : __fadd_rn(y.v[j], t);
        }
    }
    return y;
}

template <typename Tin>
__device__ __forceinline__ void reduce_vec_ieee(float (&y)[Elem<Tin>::kVec], const uint4* base, int64_t stride,
                                                int64_t v, int world, float wf, bool ok) {
    const VecF<Elem<Tin>::kVec> r = reduce_vec_ieee_out<Tin>(base, stride, v, world, wf, ok);
#pragma unroll
    for (int j = 0; j < Elem<Tin>::kVec; ++j) y[j] = r.v[j];
}

template <typename Tin>
__device__ __forceinline__ void reduce_vec_ieee_smem(float (&y)[Elem<Tin>::kVec], const unsigned char* tile,
                                                     size_t row_bytes, int world, float wf) {
    constexpr int VEC = Elem<Tin>::kVec;
#pragma unroll 1
    for (int r = 0; r < world; ++r) {
        float f[VEC];
        unpack<Tin>(*reinterpret_cast<const uint4*>(tile + (size_t)r * row_bytes), f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float t = __fdiv_rn(f[j], wf);
            y[j] = r == 0 ? t : __fadd_rn(y[j], t);
        }
    }
}

// One element on the scalar path (heads, tails, tasks that are not co-aligned).
template <typename Tin, typename Tout, int MODE, typename Args>
__device__ void flush_element(const Args& a, const TaskDesc& T, int64_t k) {
    const FlushHeader& h = a.h;
    if (!access_ok(k >= 0 && k < T.numel && T.src_off + k < h.ld, h.err)) return;
    const Tin* x = static_cast<const Tin*>(h.grads) + T.src_off + k;
    float y = 0.0f;
    for (int r = 0; r < h.world; ++r) {
        float t = pre_divide(Elem<Tin>::load(x + (int64_t)r * h.ld), MODE, h.wf, h.inv_w);
        y = (r == 0) ? t : __fadd_rn(y, t);
    }
    for (int d = 0; d < T.ndst; ++d) Elem<Tout>::store(static_cast<Tout*>(plan_dst(a, T.dst_begin + d)) + k, y);
}

// Vector body of one work unit: vectors [v0, v1) of the task's aligned body.
template <int W_T, int BATCH, typename Tin, typename Tout, int MODE, typename Args>
__device__ __forceinline__ void flush_unit_vec(const Args& a, const TaskDesc& T, int64_t v0, int64_t v1) {
    constexpr int VEC = Elem<Tin>::kVec;
    const FlushHeader& h = a.h;
    const int64_t stride = h.ld / VEC;  // row stride in vectors
    const uint4* base = reinterpret_cast<const uint4*>(static_cast<const Tin*>(h.grads) + T.src_off + T.head);
    const int64_t nbody = (T.numel - T.head) / VEC;  // used by the checks only
#pragma unroll 1
    for (int64_t vb = v0 + threadIdx.x; vb < v1; vb += (int64_t)kFlushThreads * BATCH) {
        float y[BATCH][VEC];
        // Out-of-range vectors of the last pass re-read vector vb (always in
        // range) instead of branching, and are not stored.
        int64_t vv[BATCH];
        bool ok[BATCH], tiny[BATCH];
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            vv[b] = vb + (int64_t)b * kFlushThreads < v1 ? vb + (int64_t)b * kFlushThreads : vb;
            ok[b] = access_ok(vv[b] >= 0 && vv[b] < nbody && T.src_off + T.head + (vv[b] + 1) * VEC <= h.ld, h.err);
            tiny[b] = false;
        }
        if constexpr (W_T > 0) {
            uint4 q[W_T][BATCH];
#pragma unroll
            for (int b = 0; b < BATCH; ++b)
#pragma unroll
                for (int r = 0; r < W_T; ++r) q[r][b] = load_vec(base + r * stride + vv[b], ok[b]);
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
#pragma unroll
                for (int r = 0; r < W_T; ++r) fold<Tin, MODE>(y[b], q[r][b], r == 0, h, tiny[b]);
            }
        } else {
            // Any world size: whole chunks of 8 rows (kGenericLarge only) and
            // of 4 rows, each keeping its loads in flight together, then the
            // remaining rows one at a time, all folded in rank order.
            int r0 = 0;
            if constexpr (W_T == kGenericLarge) {
#pragma unroll 1
                for (; r0 + 8 <= h.world; r0 += 8) {
                    uint4 q[8][BATCH];
#pragma unroll
                    for (int r = 0; r < 8; ++r)
#pragma unroll
                        for (int b = 0; b < BATCH; ++b)
                            q[r][b] = load_vec(base + (int64_t)(r0 + r) * stride + vv[b], ok[b]);
#pragma unroll
                    for (int b = 0; b < BATCH; ++b)
#pragma unroll
                        for (int r = 0; r < 8; ++r) fold<Tin, MODE>(y[b], q[r][b], r0 + r == 0, h, tiny[b]);
                }
            }
#pragma unroll 1
            for (; r0 + 4 <= h.world; r0 += 4) {
                uint4 q[4][BATCH];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) q[r][b] = load_vec(base + (int64_t)(r0 + r) * stride + vv[b], ok[b]);
#pragma unroll
                for (int b = 0; b < BATCH; ++b)
#pragma unroll
                    for (int r = 0; r < 4; ++r) fold<Tin, MODE>(y[b], q[r][b], r0 + r == 0, h, tiny[b]);
            }
#pragma unroll 1
            for (; r0 < h.world; ++r0) {
                uint4 q[BATCH];
#pragma unroll
                for (int b = 0; b < BATCH; ++b) q[b] = load_vec(base + (int64_t)r0 * stride + vv[b], ok[b]);
#pragma unroll
                for (int b = 0; b < BATCH; ++b) fold<Tin, MODE>(y[b], q[b], r0 == 0, h, tiny[b]);
            }
        }
        if constexpr (MODE == PDIV_DIV) {
#pragma unroll
            for (int b = 0; b < BATCH; ++b)
                if (tiny[b]) reduce_vec_ieee<Tin>(y[b], base, stride, vv[b], h.world, h.wf, ok[b]);
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            int64_t v = vb + (int64_t)b * kFlushThreads;
            const int64_t e = T.head + v * VEC;  // element index inside the task
            if (v < v1 && access_ok(e >= 0 && e + VEC <= T.numel, h.err)) {
                for (int d = 0; d < T.ndst; ++d)
                    store_vec<Tout, VEC>(static_cast<Tout*>(plan_dst(a, T.dst_begin + d)) + e, y[b]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Realigned vector path: the task's destinations are not co-aligned with its
// source (same element type, destination start shifted by sigma elements
// against the 16-byte grid of the source).  Loads stay source-aligned; each
// thread packs its vector v, takes vector v-1's packed result from the lane
// to its left (lane 0 recomputes it), and stores the destination-aligned
// 16 bytes made of the last sigma elements of v-1 and the first VEC-sigma of v.

template <typename T>
__device__ __forceinline__ uint4 pack_vec(const float (&y)[Elem<T>::kVec]);
template <>
__device__ __forceinline__ uint4 pack_vec<__nv_bfloat16>(const float (&y)[8]) {
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}
template <>
__device__ __forceinline__ uint4 pack_vec<float>(const float (&y)[4]) {
    return make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]), __float_as_uint(y[3]));
}

// Elements [VEC - S, 2 VEC - S) of the element stream P ++ C (S in 1..VEC-1).
template <typename T, int S>
__device__ __forceinline__ uint4 shifted(const uint4& P, const uint4& C) {
    const uint32_t E[8] = {P.x, P.y, P.z, P.w, C.x, C.y, C.z, C.w};
    uint32_t w[4];
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        constexpr int o = 8 - S;  // element offset, two elements per word
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (o % 2 == 0)
                w[i] = E[o / 2 + i];
            else
                w[i] = __byte_perm(E[o / 2 + i], E[o / 2 + i + 1], 0x5432);
        }
    } else {
        constexpr int o = 4 - S;  // one element per word
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = E[o + i];
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__device__ __forceinline__ uint4 shifted_rt(int s, const uint4& P, const uint4& C) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        switch (s) {
            case 1: return shifted<T, 1>(P, C);
            case 2: return shifted<T, 2>(P, C);
            case 3: return shifted<T, 3>(P, C);
            case 4: return shifted<T, 4>(P, C);
            case 5: return shifted<T, 5>(P, C);
            case 6: return shifted<T, 6>(P, C);
            default: return shifted<T, 7>(P, C);
        }
    } else {
        switch (s) {
            case 1: return shifted<T, 1>(P, C);
            case 2: return shifted<T, 2>(P, C);
            default: return shifted<T, 3>(P, C);
        }
    }
}

// Reduced, packed source vector v of the task (rows in rank order).
template <int W_T, typename T, int MODE>
__device__ __forceinline__ uint4 reduce_packed(const uint4* base, int64_t stride, int64_t v, const FlushHeader& h,
                                               bool ok) {
    constexpr int VEC = Elem<T>::kVec;
    float y[VEC];
    bool tiny = false;
    if constexpr (W_T > 0) {
        uint4 q[W_T];
#pragma unroll
        for (int r = 0; r < W_T; ++r) q[r] = load_vec(base + r * stride + v, ok);
#pragma unroll
        for (int r = 0; r < W_T; ++r) fold<T, MODE>(y, q[r], r == 0, h, tiny);
    } else {
        for (int r = 0; r < h.world; ++r) fold<T, MODE>(y, load_vec(base + (int64_t)r * stride + v, ok), r == 0, h, tiny);
    }
    if constexpr (MODE == PDIV_DIV)
        if (tiny) reduce_vec_ieee<T>(y, base, stride, v, h.world, h.wf, ok);
    return pack_vec<T>(y);
}

// Barrier over the kFlushThreads threads that reduce (id 1; in the TMA kernel
// the producer thread never reaches it).
__device__ __forceinline__ void reducers_barrier() {
    asm volatile("bar.sync 1, %0;" ::"r"(kFlushThreads) : "memory");
}

// Vectors [v0, v1) of the task's source body, one per thread per pass.  A
// thread takes vector v-1's packed result from the lane to its left, lane 0
// of a warp from lane 31 of the warp before it (shared memory), and thread 0
// from the last thread of the previous pass.  The output that straddles the
// unit's first vector and the previous unit is written on the scalar path by
// the caller.  Passes are uniform across the block so that every thread takes
// part in the shuffles and barriers; out-of-range threads re-read vector v1-1
// and store nothing.
template <int W_T, typename T, int MODE, typename Args>
__device__ __forceinline__ void flush_unit_realign(const Args& a, const TaskDesc& Tk, int64_t v0, int64_t v1,
                                                   int sigma) {
    constexpr int VEC = Elem<T>::kVec;
    __shared__ uint4 s_last[kFlushThreads / 32];
    __shared__ uint4 s_carry;
    const FlushHeader& h = a.h;
    const int64_t stride = h.ld / VEC;
    const uint4* base = reinterpret_cast<const uint4*>(static_cast<const T*>(h.grads) + Tk.src_off + Tk.head);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int64_t pb = v0; pb < v1; pb += kFlushThreads) {
        const int64_t v = pb + t;
        const int64_t vl = v < v1 ? v : v1 - 1;
        const bool ok = access_ok(vl >= 0 && vl < (Tk.numel - Tk.head) / VEC &&
                                      Tk.src_off + Tk.head + (vl + 1) * VEC <= h.ld, h.err);
        const uint4 C = reduce_packed<W_T, T, MODE>(base, stride, vl, h, ok);
        uint4 P;
        P.x = __shfl_up_sync(0xffffffffu, C.x, 1);
        P.y = __shfl_up_sync(0xffffffffu, C.y, 1);
        P.z = __shfl_up_sync(0xffffffffu, C.z, 1);
        P.w = __shfl_up_sync(0xffffffffu, C.w, 1);
        if (lane == 31) s_last[warp] = C;
        reducers_barrier();
        if (lane == 0) P = warp > 0 ? s_last[warp - 1] : s_carry;  // s_carry: set by the previous pass
        reducers_barrier();
        if (t == kFlushThreads - 1) s_carry = C;
        const int64_t e = Tk.head + v * VEC - sigma;  // destination-aligned element index
        if (v > v0 && v < v1 && access_ok(e >= 0 && e + VEC <= Tk.numel, h.err)) {
            const uint4 out = shifted_rt<T>(sigma, P, C);
            for (int d = 0; d < Tk.ndst; ++d)
                __stcs(reinterpret_cast<uint4*>(static_cast<T*>(plan_dst(a, Tk.dst_begin + d)) + e), out);
        }
    }
}

// Unit of a realigned task: its vectors, plus (in unit 0) the scalar head
// [0, head + VEC - sigma) and tail [head + VEC * nbody - sigma, numel).
template <int W_T, typename Tin, typename Tout, int MODE, typename Args>
__device__ __forceinline__ void flush_unit_shifted(const Args& a, const TaskDesc& T, int64_t local, int threads) {
    if constexpr (std::is_same<Tin, Tout>::value) {
        constexpr int VEC = Elem<Tin>::kVec;
        const int sigma = T.vec - 1;
        const int64_t nbody = (T.numel - T.head) / VEC;
        const int64_t v0 = local * (int64_t)a.h.unit_vec;
        const int64_t v1 = v0 + a.h.unit_vec < nbody ? v0 + a.h.unit_vec : nbody;
        flush_unit_realign<W_T, Tin, MODE>(a, T, v0, v1, sigma);
        // the destination vector that straddles vector v0-1 and v0 (another unit)
        if (v0 >= 1 && (int)threadIdx.x < VEC) flush_element<Tin, Tout, MODE>(a, T, T.head + v0 * VEC - sigma + threadIdx.x);
        if (local == 0) {
            const int hcount = T.head + VEC - sigma;
            const int64_t tstart = T.head + nbody * VEC - sigma;
            const int tcount = (int)(T.numel - tstart);
            for (int id = threadIdx.x; id < hcount + tcount; id += threads)
                flush_element<Tin, Tout, MODE>(a, T, id < hcount ? id : tstart + (id - hcount));
        }
    }
}

template <int W_T, int BATCH, typename Tin, typename Tout, int MODE, bool RA, typename Args>
__device__ __forceinline__ void flush_unit(const Args& a, const TaskDesc& T, int64_t local) {
    constexpr int VEC = Elem<Tin>::kVec;
    if (RA && T.vec >= 2) {
        if constexpr (RA) flush_unit_shifted<W_T, Tin, Tout, MODE>(a, T, local, kFlushThreads);
    } else if (T.vec) {
        const int64_t nbody = (T.numel - T.head) / VEC;
        const int64_t v0 = local * h_unit(a);
        const int64_t v1 = v0 + h_unit(a) < nbody ? v0 + h_unit(a) : nbody;
        flush_unit_vec<W_T, BATCH, Tin, Tout, MODE>(a, T, v0, v1);
        if (local == 0) {
            const int tail = (int)(T.numel - T.head - nbody * VEC);
            const int id = threadIdx.x;
            if (id < T.head)
                flush_element<Tin, Tout, MODE>(a, T, id);
            else if (id < T.head + tail)
                flush_element<Tin, Tout, MODE>(a, T, T.head + nbody * VEC + (id - T.head));
        }
    } else {
        const int64_t e0 = local * kUnitScalar;
        const int64_t e1 = e0 + kUnitScalar < T.numel ? e0 + kUnitScalar : T.numel;
        for (int64_t k = e0 + threadIdx.x; k < e1; k += kFlushThreads) flush_element<Tin, Tout, MODE>(a, T, k);
    }
}

// The plan task that work unit u belongs to: the last task whose first unit is <= u.
template <typename Args>
__device__ __forceinline__ int find_task(const Args& a, int64_t u) {
    int lo = 0, hi = a.h.n_tasks - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (plan_task(a, mid).unit_begin <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// RA: the plan holds realigned tasks (destinations shifted against the
// source).  That path is compiled into its own kernel so that the common
// kernel keeps its register budget.
//
// Programmatic dependent launch: every CTA lets the next launch on the stream
// start as soon as it is running, and waits for the previous launch's grid
// to complete before it exits.  A flush launched with programmatic stream
// serialisation (only ever one whose bucket shares no byte with the previous
// one) therefore fills the SMs that the previous flush's last wave leaves
// idle, and still completes after it, so the stream's order of completion is
// unchanged.  Launched without the attribute, both instructions do nothing.
template <int W_T, int BATCH, typename Tin, typename Tout, typename Args, bool RA>
__global__ void __launch_bounds__(kFlushThreads, flush_min_blocks(W_T)) flush_kernel(const __grid_constant__ Args a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const FlushHeader& h = a.h;
    for (int64_t u = blockIdx.x; u < h.total_units; u += gridDim.x) {
        const TaskDesc T = plan_task(a, find_task(a, u));
        const int64_t local = u - T.unit_begin;
        // a power-of-two world size never divides (its pre-division is the
        // exact multiply), so its kernels carry no division path at all
        if (h.pdiv == PDIV_POW2)
            flush_unit<W_T, BATCH, Tin, Tout, PDIV_POW2, RA>(a, T, local);
        else if (may_divide(W_T) && h.pdiv == PDIV_DIV)
            flush_unit<W_T, BATCH, Tin, Tout, div_mode<Tin>(W_T), RA>(a, T, local);
        else
            flush_unit<W_T, BATCH, Tin, Tout, PDIV_NONE, RA>(a, T, local);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA-staged flush.  One producer thread per CTA streams the W row tiles of
// every sub-tile (kSubVec 16-byte vectors = 4 KB per row) into a ring of
// shared-memory stages with cp.async.bulk, each stage's arrival counted on its
// `full` mbarrier; eight consumer warps reduce a stage from shared memory (one
// vector per thread, rank order), store the result to the delivered
// destinations and release the stage on its `empty` mbarrier.  The ring keeps
// up to 192 KB of every SM's share of the bucket in flight without holding it
// in registers.  Scalar work (heads, tails, tasks that are not co-aligned) is
// done by the consumers straight from global memory, as in flush_kernel.
// ---------------------------------------------------------------------------

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kTmaThreads = kTmaConsumers + 32;
constexpr int kSubVec = 256;                  // 16-byte vectors per row per stage
constexpr uint32_t kTmaRowBytes = kSubVec * 16;
constexpr int kTmaStageBudget = 192 * 1024;   // shared memory given to the stage ring

template <int W>
__host__ __device__ constexpr int tma_stages() {
    constexpr int s = kTmaStageBudget / (W * (int)kTmaRowBytes);
    return s > 16 ? 16 : (s < 2 ? 2 : s);
}

template <int W>
__host__ __device__ constexpr size_t tma_smem_bytes() {
    return (size_t)tma_stages<W>() * W * kTmaRowBytes;
}

template <int W_T, typename Tin, typename Tout, int MODE, typename Args>
__device__ void tma_consume(const Args& a, unsigned char* smem, uint64_t* full, uint64_t* empty, int* abort_flag) {
    constexpr int VEC = Elem<Tin>::kVec;
    constexpr int STAGES = tma_stages<W_T>();
    const FlushHeader& h = a.h;
    const int ctid = threadIdx.x, lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = blockIdx.x; u < h.total_units; u += gridDim.x) {
        const TaskDesc T = plan_task(a, find_task(a, u));
        const int64_t local = u - T.unit_begin;
        if (!T.vec) {
            const int64_t e0 = local * kUnitScalar;
            const int64_t e1 = e0 + kUnitScalar < T.numel ? e0 + kUnitScalar : T.numel;
            for (int64_t k = e0 + ctid; k < e1; k += kTmaConsumers) flush_element<Tin, Tout, MODE>(a, T, k);
            continue;
        }
        if (T.vec >= 2) {  // destinations shifted against the source: register path, no staging
            flush_unit_shifted<W_T, Tin, Tout, MODE>(a, T, local, kTmaConsumers);
            continue;
        }
        const int64_t nbody = (T.numel - T.head) / VEC;
        const int64_t v0 = local * (int64_t)h.unit_vec;
        const int64_t v1 = v0 + h.unit_vec < nbody ? v0 + h.unit_vec : nbody;
        if (local == 0) {
            const int tail = (int)(T.numel - T.head - nbody * VEC);
            if (ctid < T.head)
                flush_element<Tin, Tout, MODE>(a, T, ctid);
            else if (ctid < T.head + tail)
                flush_element<Tin, Tout, MODE>(a, T, T.head + nbody * VEC + (ctid - T.head));
        }
        for (int64_t sv = v0; sv < v1; sv += kSubVec) {
            const int64_t nv = v1 - sv < kSubVec ? v1 - sv : kSubVec;
            if (!tma::mbar_wait(&full[stage], phase)) {
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                record_device_error(h.err, DPRED_E_TIMEOUT);
                return;
            }
            if (ctid < nv) {
                const unsigned char* tile = smem + (size_t)stage * W_T * kTmaRowBytes + (size_t)ctid * 16;
                float y[VEC];
                bool tiny = false;
#pragma unroll
                for (int r = 0; r < W_T; ++r) {
                    const uint4 q = *reinterpret_cast<const uint4*>(tile + (size_t)r * kTmaRowBytes);
                    fold<Tin, MODE>(y, q, r == 0, h, tiny);
                }
                if constexpr (MODE == PDIV_DIV)
                    if (tiny) reduce_vec_ieee_smem<Tin>(y, tile, kTmaRowBytes, W_T, h.wf);
                const int64_t e = T.head + (sv + ctid) * VEC;
                if (access_ok(e >= 0 && e + VEC <= T.numel, h.err))
                    for (int d = 0; d < T.ndst; ++d)
                        store_vec<Tout, VEC>(static_cast<Tout*>(plan_dst(a, T.dst_begin + d)) + e, y);
            }
            __syncwarp();
            if (lane == 0) tma::mbar_arrive(&empty[stage]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
}

template <int W_T, typename Tin, typename Tout, typename Args>
__device__ void tma_produce(const Args& a, unsigned char* smem, uint64_t* full, uint64_t* empty, int* abort_flag) {
    constexpr int VEC = Elem<Tin>::kVec;
    constexpr int STAGES = tma_stages<W_T>();
    const FlushHeader& h = a.h;
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; ok && u < h.total_units; u += gridDim.x) {
        const TaskDesc T = plan_task(a, find_task(a, u));
        if (T.vec != 1) continue;  // only co-aligned vector tasks are staged
        const int64_t local = u - T.unit_begin;
        const int64_t nbody = (T.numel - T.head) / VEC;
        const int64_t v0 = local * (int64_t)h.unit_vec;
        const int64_t v1 = v0 + h.unit_vec < nbody ? v0 + h.unit_vec : nbody;
        const char* base = reinterpret_cast<const char*>(static_cast<const Tin*>(h.grads) + T.src_off + T.head);
        const int64_t row_bytes = h.ld * (int64_t)sizeof(Tin);
        for (int64_t sv = v0; sv < v1; sv += kSubVec) {
            const uint32_t bytes = (uint32_t)((v1 - sv < kSubVec ? v1 - sv : kSubVec) * 16);
            if (*reinterpret_cast<volatile int*>(abort_flag) || !tma::mbar_wait(&empty[stage], phase ^ 1)) {
                ok = false;
                break;
            }
            // a checked build that rejects the range completes the stage with no bytes
            const bool in = access_ok(sv >= 0 && (sv * 16 + bytes) <= nbody * 16 &&
                                          T.src_off + T.head + (sv * 16 + bytes) / (int64_t)sizeof(Tin) <= h.ld,
                                      h.err);
            tma::mbar_arrive_expect_tx(&full[stage], in ? bytes * W_T : 0u);
            if (in) {
#pragma unroll
                for (int r = 0; r < W_T; ++r)
                    tma::bulk_load(smem + ((size_t)stage * W_T + r) * kTmaRowBytes, base + r * row_bytes + sv * 16,
                                   bytes, &full[stage]);
            }
            ++issued;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    if (!ok) record_device_error(h.err, DPRED_E_TIMEOUT);
    // Leave only after every bulk copy this thread issued has landed.
    const int64_t pend = issued < STAGES ? issued : STAGES;
    for (int64_t q = issued - pend; q < issued; ++q)
        if (!tma::mbar_wait(&full[q % STAGES], (uint32_t)((q / STAGES) & 1))) {
            record_device_error(h.err, DPRED_E_TIMEOUT);
            break;
        }
}

template <int W_T, typename Tin, typename Tout, typename Args>
__global__ void __launch_bounds__(kTmaThreads, 1) flush_tma_kernel(const __grid_constant__ Args a) {
    constexpr int STAGES = tma_stages<W_T>();
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ __align__(8) uint64_t empty[STAGES];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tma::mbar_init(&full[s], 1);
            tma::mbar_init(&empty[s], kTmaConsumerWarps);
        }
        abort_flag = 0;
        tma::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x >= kTmaConsumers) {
        if (threadIdx.x == kTmaConsumers) tma_produce<W_T, Tin, Tout>(a, smem, full, empty, &abort_flag);
        return;
    }
    const int mode = a.h.pdiv;
    if (mode == PDIV_POW2)
        tma_consume<W_T, Tin, Tout, PDIV_POW2>(a, smem, full, empty, &abort_flag);
    else if (may_divide(W_T) && mode == PDIV_DIV)
        tma_consume<W_T, Tin, Tout, div_mode<Tin>(W_T)>(a, smem, full, empty, &abort_flag);
    else
        tma_consume<W_T, Tin, Tout, PDIV_NONE>(a, smem, full, empty, &abort_flag);
}

// Persistent grid: SMs x resident CTAs of this kernel, capped by the number of units.
template <typename K>
int64_t persistent_grid(K kernel, int64_t units, int max_per_sm) {
    int occ = resident_ctas(reinterpret_cast<const void*>(kernel), kFlushThreads);
    if (occ > max_per_sm) occ = max_per_sm;
    int64_t g = (int64_t)sm_count() * occ;
    return units < g ? units : g;
}

// One launch of the LDG kernel (any W) or, for W in {2, 4, 8, 16} when the
// TMA path is selected, of the TMA-staged kernel (one CTA per SM).  Plans that
// touch host memory always take the LDG kernel: its plain loads and stores
// reach pinned host memory over the host link, and no bulk copy is issued there.
// Launch of the LDG kernel, with programmatic stream serialisation when pdl.
// per_unit: the kernel may launch one CTA per work unit (flush_grid_per_unit).
// It does so unless the launch overlaps the previous one (pdl) and has fewer
// than 8 units per CTA of the persistent grid: a short overlapped flush gains
// more from starting on the previous flush's idle SMs, which a persistent grid
// does at once, than from the block scheduler's balance.  Sweep A/B, fraction
// of the copy peak, persistent -> one CTA per unit, consecutive overlapped
// calls: W = 16, 4 MB per replica 1.045 -> 0.975; W = 24 fp32, 16 MB 1.006 ->
// 0.935; the same launches without the overlap promise: 0.778 -> 0.766 and
// 0.645 -> 0.810.
template <typename K, typename Args>
cudaError_t launch_ldg(K k, const Args& a, int64_t units, int max_per_sm, bool per_unit, bool pdl, cudaStream_t s) {
    const int64_t pg = persistent_grid(k, units, max_per_sm);
    const bool one_per_unit = per_unit && (!pdl || units >= 8 * pg);
    const unsigned grid = one_per_unit ? (unsigned)(units < 0x7FFFFFFF ? units : 0x7FFFFFFF) : (unsigned)pg;
    if (!pdl) {
        k<<<grid, kFlushThreads, 0, s>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFlushThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <int W_T, int BATCH, typename Tin, typename Tout, typename Args>
cudaError_t launch_kernel(const Args& a, int64_t units, bool realign, bool ldg_only, bool write_heavy, bool pdl,
                          cudaStream_t s) {
    const int cap = flush_ctas_per_sm(W_T, write_heavy);
    if constexpr (W_T == 2 || W_T == 4 || W_T == 8 || W_T == 16) {  // the TMA form's world sizes
        if (!ldg_only && flush_path() == PATH_TMA) {  // auto: the register-streaming form measured faster on GB300
            auto k = flush_tma_kernel<W_T, Tin, Tout, Args>;
            constexpr size_t smem = tma_smem_bytes<W_T>();
            static bool attr[64] = {};
            cudaError_t ea = ensure_smem_attr(k, (int)smem, attr);
            if (ea != cudaSuccess) return ea;
            int64_t g = sm_count();
            k<<<(unsigned)(units < g ? units : g), kTmaThreads, smem, s>>>(a);
            return cudaGetLastError();
        }
    }
    const bool per_unit = flush_grid_per_unit(W_T, a.h.pdiv == PDIV_POW2);
    if constexpr (std::is_same<Tin, Tout>::value) {
        if (realign)
            return launch_ldg(flush_kernel<W_T, BATCH, Tin, Tout, Args, true>, a, units, cap, per_unit, pdl, s);
    }
    return launch_ldg(flush_kernel<W_T, BATCH, Tin, Tout, Args, false>, a, units, cap, per_unit, pdl, s);
}

template <int W_T, int BATCH, typename Tin, typename Tout>
int launch_flush_w(const FlushLaunch& L, cudaStream_t s) {
    static_assert(BATCH == flush_batch_of(W_T, std::is_same<Tin, __nv_bfloat16>::value),
                  "one batch per world size and input type");
    const FlushHeader& h = L.h;
    if (h.total_units == 0) return DPRED_OK;
    cudaError_t e;
    if (h.n_tasks <= kInlineTasks && L.n_dst <= kInlineDst) {
        FlushArgsInline a;
        a.h = h;
        for (int i = 0; i < h.n_tasks; ++i) a.tasks[i] = L.tasks[i];
        for (int i = 0; i < L.n_dst; ++i) a.dst[i] = L.dst[i];
        e = launch_kernel<W_T, BATCH, Tin, Tout>(a, h.total_units, L.realign, L.ldg_only, L.write_heavy, L.pdl, s);
    } else {
        size_t tb = sizeof(TaskDesc) * (size_t)h.n_tasks, db = sizeof(void*) * (size_t)L.n_dst;
        size_t need = tb + ((db + 15) & ~(size_t)15);
        if (L.workspace == nullptr || L.workspace_bytes < need)
            return set_error(DPRED_E_SIZE, "flush plan of %d tasks / %d destinations needs %zu bytes of workspace, got %zu",
                             h.n_tasks, L.n_dst, need, L.workspace_bytes);
        if ((reinterpret_cast<uintptr_t>(L.workspace) & 15) != 0)
            return set_error(DPRED_E_ALIGN, "flush workspace must be 16-byte aligned");
        const int rc = refuse_capture_of_upload(s, "a flush plan");
        if (rc != DPRED_OK) return rc;
        char* ws = static_cast<char*>(L.workspace);
        e = cudaMemcpyAsync(ws, L.tasks, tb, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess && db) e = cudaMemcpyAsync(ws + tb, L.dst, db, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_error(e, "flush plan copy");
        FlushArgsWs a;
        a.h = h;
        a.tasks = reinterpret_cast<const TaskDesc*>(ws);
        a.dst = reinterpret_cast<void* const*>(ws + tb);
        // the plan upload sits between this launch and the previous one: no overlap
        e = launch_kernel<W_T, BATCH, Tin, Tout>(a, h.total_units, L.realign, L.ldg_only, L.write_heavy, false, s);
    }
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "flush kernel launch");
}

// Each world size's launchers are compiled in a translation unit of their
// own (flush_w*.cu, one DPRED_FLUSH_INSTANTIATE line each) so that nvcc builds
// them in parallel; the dispatcher sees them as extern templates.
#define DPRED_FLUSH_W_FOR_TYPES(X, W)                                                         \
    X(W, dpred::flush_batch_of(W, true), __nv_bfloat16, __nv_bfloat16)                       \
    X(W, dpred::flush_batch_of(W, true), __nv_bfloat16, float)                               \
    X(W, dpred::flush_batch_of(W, false), float, float)                                      \
    X(W, dpred::flush_batch_of(W, false), float, __nv_bfloat16)
#define DPRED_FLUSH_INSTANTIATE_ONE(W, B, Tin, Tout) \
    template int dpred::launch_flush_w<W, B, Tin, Tout>(const dpred::FlushLaunch&, cudaStream_t);
#define DPRED_FLUSH_DECLARE_ONE(W, B, Tin, Tout) \
    extern template int dpred::launch_flush_w<W, B, Tin, Tout>(const dpred::FlushLaunch&, cudaStream_t);
#define DPRED_FLUSH_INSTANTIATE(W) DPRED_FLUSH_W_FOR_TYPES(DPRED_FLUSH_INSTANTIATE_ONE, W)
#define DPRED_FLUSH_DECLARE(W) DPRED_FLUSH_W_FOR_TYPES(DPRED_FLUSH_DECLARE_ONE, W)
// bf16 inputs only (the generic loop for many ranks).
#define DPRED_FLUSH_W_FOR_BF16_IN(X, W)                                                        \
    X(W, dpred::flush_batch_of(W, true), __nv_bfloat16, __nv_bfloat16)                       \
    X(W, dpred::flush_batch_of(W, true), __nv_bfloat16, float)
#define DPRED_FLUSH_INSTANTIATE_BF16_IN(W) DPRED_FLUSH_W_FOR_BF16_IN(DPRED_FLUSH_INSTANTIATE_ONE, W)
#define DPRED_FLUSH_DECLARE_BF16_IN(W) DPRED_FLUSH_W_FOR_BF16_IN(DPRED_FLUSH_DECLARE_ONE, W)

}  // namespace dpred
