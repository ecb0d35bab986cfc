// accumulate.cu -- replica-local gradient accumulation and the one cross-replica
// reduction per optimizer step.
//
// MaxText PR #5099 "Defer the data-parallel gradient all-reduce to update()
// under gradient accumulation", section "What": cotangents stay per-replica
// partial sums that accumulate replica-locally across micro-batches, and the
// single cross-replica all-reduce happens once, in update().  Here the W
// replica accumulators are rows of one [W, n] fp32 array; a micro-batch adds
// its [W, n] gradient row by row (acc += g), and the last micro-batch's add is
// fused with the reduction over rows (total = sum_r (acc_r + g_r)), so the
// accumulator is read once and never written back on that pass.
#include <type_traits>

#include "common.cuh"

namespace dpred {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Streaming loads of acc and g.  With fp32 gradients they are cached in L2
// only (ld.global.cg); with bf16 gradients they are evict-first
// (ld.global.cs).  Interleaved A/B on GB300: .cg made the fp32 W=4 add 0.9%
// faster (0.981 -> 0.990 of the copy peak) and the bf16 W=8 add 0.2% slower;
// the finalize pass was equal.
template <typename Tg, typename V>
__device__ __forceinline__ V acc_ld(const V* p) {
    if constexpr (std::is_same<Tg, float>::value)
        return __ldcg(p);
    else
        return __ldcs(p);
}

template <typename Tg>
struct G;
template <>
struct G<__nv_bfloat16> {
    using V = uint2;  // 4 bf16
    __device__ static void widen(const V& v, float (&f)[4]) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    }
    __device__ static float one(const __nv_bfloat16* p) { return bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(p)); }
};
template <>
struct G<float> {
    using V = float4;
    __device__ static void widen(const V& v, float (&f)[4]) { f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w; }
    __device__ static float one(const float* p) { return *p; }
};

// acc[i] = first ? g[i] : acc[i] + g[i] over the flat [W * n] range.
template <typename Tg, bool FIRST>
__global__ void __launch_bounds__(kThreads) accumulate_kernel(float* __restrict__ acc, const Tg* __restrict__ g,
                                                              int64_t total, int vec) {
    using V = typename G<Tg>::V;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = total / 4;
        float4* a4 = reinterpret_cast<float4*>(acc);
        const V* g4 = reinterpret_cast<const V*>(g);
        for (int64_t v0 = tid; v0 < nv; v0 += nthreads * kUnroll) {
            float4 av[kUnroll];
            V gv[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int64_t v = v0 + u * nthreads;
                if (v < nv) {
                    if (!FIRST) av[u] = acc_ld<Tg>(a4 + v);
                    gv[u] = acc_ld<Tg>(g4 + v);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int64_t v = v0 + u * nthreads;
                if (v < nv) {
                    float f[4];
                    G<Tg>::widen(gv[u], f);
                    float4 o;
                    if (FIRST) {
                        o = make_float4(f[0], f[1], f[2], f[3]);
                    } else {
                        o = make_float4(__fadd_rn(av[u].x, f[0]), __fadd_rn(av[u].y, f[1]), __fadd_rn(av[u].z, f[2]),
                                        __fadd_rn(av[u].w, f[3]));
                    }
                    __stcs(a4 + v, o);
                }
            }
        }
        done = nv * 4;
    }
    for (int64_t i = done + tid; i < total; i += nthreads) {
        float gv = G<Tg>::one(g + i);
        acc[i] = FIRST ? gv : __fadd_rn(acc[i], gv);
    }
}

// total[k] = (sum over r in order of (first ? g[r][k] : acc[r][k] + g[r][k])) * scale.
template <int W_T, typename Tg, bool FIRST>
__global__ void __launch_bounds__(kThreads) finalize_kernel(const float* __restrict__ acc, const Tg* __restrict__ g,
                                                            float* __restrict__ total, int world, int64_t n,
                                                            float scale, int vec) {
    using V = typename G<Tg>::V;
    const int W = W_T > 0 ? W_T : world;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n / 4;
        const float4* a4 = reinterpret_cast<const float4*>(acc);
        const V* g4 = reinterpret_cast<const V*>(g);
        float4* t4 = reinterpret_cast<float4*>(total);
        for (int64_t v = tid; v < nv; v += nthreads) {
            float y[4];
            if constexpr (W_T > 0) {
                float4 av[W_T];
                V gv[W_T];
#pragma unroll
                for (int r = 0; r < W_T; ++r) {
                    if (!FIRST) av[r] = acc_ld<Tg>(a4 + r * nv + v);
                    gv[r] = acc_ld<Tg>(g4 + r * nv + v);
                }
#pragma unroll
                for (int r = 0; r < W_T; ++r) {
                    float f[4];
                    G<Tg>::widen(gv[r], f);
                    float a[4] = {f[0], f[1], f[2], f[3]};
                    if (!FIRST) {
                        a[0] = __fadd_rn(av[r].x, f[0]); a[1] = __fadd_rn(av[r].y, f[1]);
                        a[2] = __fadd_rn(av[r].z, f[2]); a[3] = __fadd_rn(av[r].w, f[3]);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) y[j] = (r == 0) ? a[j] : __fadd_rn(y[j], a[j]);
                }
            } else {
                for (int r = 0; r < W; ++r) {
                    float f[4];
                    G<Tg>::widen(acc_ld<Tg>(g4 + r * nv + v), f);
                    if (!FIRST) {
                        float4 av = acc_ld<Tg>(a4 + r * nv + v);
                        f[0] = __fadd_rn(av.x, f[0]); f[1] = __fadd_rn(av.y, f[1]);
                        f[2] = __fadd_rn(av.z, f[2]); f[3] = __fadd_rn(av.w, f[3]);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) y[j] = (r == 0) ? f[j] : __fadd_rn(y[j], f[j]);
                }
            }
            __stcs(t4 + v, make_float4(__fmul_rn(y[0], scale), __fmul_rn(y[1], scale), __fmul_rn(y[2], scale),
                                       __fmul_rn(y[3], scale)));
        }
        done = nv * 4;
    }
    for (int64_t k = done + tid; k < n; k += nthreads) {
        float y = 0.0f;
        for (int r = 0; r < W; ++r) {
            float a = G<Tg>::one(g + (int64_t)r * n + k);
            if (!FIRST) a = __fadd_rn(acc[(int64_t)r * n + k], a);
            y = (r == 0) ? a : __fadd_rn(y, a);
        }
        total[k] = __fmul_rn(y, scale);
    }
}

// Resident CTAs per SM of the micro-batch add (grid cap).  Interleaved A/B on
// GB300 with the grid capped at 1, 2, 3 or 4 CTAs per SM (4 fit): 2 is best,
// 1.007 of the measured copy peak on the 402.8M W=8 bf16 add (0.788, 0.981,
// 0.973 at 1, 3, 4) and 1.008 on the qwen3 W=4 fp32 add (0.871, 0.994, 0.990).
// The finalize pass keeps full occupancy (capped at 2 it fell to 0.58).
constexpr int kAccAddCtasPerSm = 2;
template <typename K>
unsigned grid_for(K kernel, int64_t work_items, int max_per_sm = 1 << 30) {
    int occ = resident_ctas(reinterpret_cast<const void*>(kernel), kThreads);
    if (occ > max_per_sm) occ = max_per_sm;
    int64_t g = (int64_t)sm_count() * occ;
    int64_t need = (work_items + kThreads - 1) / kThreads;
    if (need < 1) need = 1;
    return (unsigned)(need < g ? need : g);
}

template <typename Tg, bool FIRST>
int launch_finalize(int world, int64_t n, const float* acc, const Tg* g, float* total, float scale, int vec,
                    cudaStream_t s) {
    int64_t items = vec ? n / 4 : n;
#define DPRED_FIN(WT)                                                                     \
    {                                                                                     \
        auto k = finalize_kernel<WT, Tg, FIRST>;                                          \
        k<<<grid_for(k, items), kThreads, 0, s>>>(acc, g, total, world, n, scale, vec);   \
        break;                                                                            \
    }
    switch (world) {
        case 1: DPRED_FIN(1)
        case 2: DPRED_FIN(2)
        case 4: DPRED_FIN(4)
        case 8: DPRED_FIN(8)
        default: DPRED_FIN(0)
    }
#undef DPRED_FIN
    return DPRED_OK;
}

template <typename Tg>
int launch_typed(int world, int64_t n, float* acc, const Tg* g, int first, int finalize, float scale, float* total,
                 cudaStream_t s) {
    const int64_t total_elems = (int64_t)world * n;
    const uintptr_t ga = reinterpret_cast<uintptr_t>(g), aa = reinterpret_cast<uintptr_t>(acc);
    const int gvec = (int)sizeof(typename G<Tg>::V);
    if (!finalize) {
        // flat over [W * n]: rows are contiguous, so only the bases need alignment
        int vec = (aa % 16 == 0) && (ga % gvec == 0);
        int64_t items = vec ? total_elems / 4 : total_elems;
        if (first) {
            auto k = accumulate_kernel<Tg, true>;
            k<<<grid_for(k, items, kAccAddCtasPerSm), kThreads, 0, s>>>(acc, g, total_elems, vec);
        } else {
            auto k = accumulate_kernel<Tg, false>;
            k<<<grid_for(k, items, kAccAddCtasPerSm), kThreads, 0, s>>>(acc, g, total_elems, vec);
        }
    } else {
        // per column: every row start must keep the vector alignment
        int vec = (aa % 16 == 0) && (ga % gvec == 0) && (n % 4 == 0) &&
                  (reinterpret_cast<uintptr_t>(total) % 16 == 0);
        if (first)
            launch_finalize<Tg, true>(world, n, acc, g, total, scale, vec, s);
        else
            launch_finalize<Tg, false>(world, n, acc, g, total, scale, vec, s);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "accumulate kernel launch");
}

// Checkpoint form of the accumulator (MaxText PR #5099, "Accumulator
// lifetime"): save reduces the replica rows to the total a checkpoint holds;
// restore writes a total back as row 0 with zeros in the other rows.
template <int W_T>
__global__ void __launch_bounds__(kThreads) save_kernel(const float* __restrict__ acc, float* __restrict__ total,
                                                        int world, int64_t n, int vec) {
    const int W = W_T > 0 ? W_T : world;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n / 4;
        const float4* a4 = reinterpret_cast<const float4*>(acc);
        float4* t4 = reinterpret_cast<float4*>(total);
        for (int64_t v = tid; v < nv; v += nthreads) {
            float4 y = __ldcs(a4 + v);
            if constexpr (W_T > 0) {
                float4 q[W_T > 1 ? W_T - 1 : 1];
#pragma unroll
                for (int r = 1; r < W_T; ++r) q[r - 1] = __ldcs(a4 + r * nv + v);
#pragma unroll
                for (int r = 1; r < W_T; ++r)
                    y = make_float4(__fadd_rn(y.x, q[r - 1].x), __fadd_rn(y.y, q[r - 1].y), __fadd_rn(y.z, q[r - 1].z),
                                    __fadd_rn(y.w, q[r - 1].w));
            } else {
                for (int r = 1; r < W; ++r) {
                    const float4 q = __ldcs(a4 + r * nv + v);
                    y = make_float4(__fadd_rn(y.x, q.x), __fadd_rn(y.y, q.y), __fadd_rn(y.z, q.z), __fadd_rn(y.w, q.w));
                }
            }
            __stcs(t4 + v, y);
        }
        done = nv * 4;
    }
    for (int64_t k = done + tid; k < n; k += nthreads) {
        float y = acc[k];
        for (int r = 1; r < W; ++r) y = __fadd_rn(y, acc[(int64_t)r * n + k]);
        total[k] = y;
    }
}

__global__ void __launch_bounds__(kThreads) restore_kernel(float* __restrict__ acc, const float* __restrict__ total,
                                                           int world, int64_t n, int vec) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    if (vec) {
        const int64_t nv = n / 4, all = (int64_t)world * nv;
        float4* a4 = reinterpret_cast<float4*>(acc);
        const float4* t4 = reinterpret_cast<const float4*>(total);
        for (int64_t i = tid; i < all; i += nthreads)
            __stcs(a4 + i, i < nv ? __ldcs(t4 + i) : make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const int64_t all = (int64_t)world * n;
    for (int64_t i = tid; i < all; i += nthreads) acc[i] = i < n ? total[i] : 0.0f;
}

}  // namespace

int launch_accumulator_save(int world, int64_t n, const float* acc, float* total, cudaStream_t s) {
    if ((int64_t)world * n == 0) return DPRED_OK;
    const int vec = reinterpret_cast<uintptr_t>(acc) % 16 == 0 && reinterpret_cast<uintptr_t>(total) % 16 == 0 &&
                    n % 4 == 0;
    const int64_t items = vec ? n / 4 : n;
#define DPRED_SAVE(WT)                                                             \
    {                                                                              \
        auto k = save_kernel<WT>;                                                  \
        k<<<grid_for(k, items), kThreads, 0, s>>>(acc, total, world, n, vec);      \
        break;                                                                     \
    }
    switch (world) {
        case 1: DPRED_SAVE(1)
        case 2: DPRED_SAVE(2)
        case 4: DPRED_SAVE(4)
        case 8: DPRED_SAVE(8)
        default: DPRED_SAVE(0)
    }
#undef DPRED_SAVE
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "accumulator save launch");
}

int launch_accumulator_restore(int world, int64_t n, float* acc, const float* total, cudaStream_t s) {
    if ((int64_t)world * n == 0) return DPRED_OK;
    const int vec = reinterpret_cast<uintptr_t>(acc) % 16 == 0 && reinterpret_cast<uintptr_t>(total) % 16 == 0 &&
                    n % 4 == 0;
    const int64_t items = vec ? (int64_t)world * n / 4 : (int64_t)world * n;
    restore_kernel<<<grid_for(restore_kernel, items), kThreads, 0, s>>>(acc, total, world, n, vec);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "accumulator restore launch");
}

int launch_accumulate(int world, int64_t n, float* acc, int g_dt, const void* g, int first, int finalize, float scale,
                      float* total, cudaStream_t s) {
    if ((int64_t)world * n == 0) return DPRED_OK;
    if (g_dt == DPRED_BF16)
        return launch_typed(world, n, acc, static_cast<const __nv_bfloat16*>(g), first, finalize, scale, total, s);
    return launch_typed(world, n, acc, static_cast<const float*>(g), first, finalize, scale, total, s);
}

}  // namespace dpred
