// owner_map.cu -- the ZeRO-1 owner map computed on the device.
//
// DeepSpeed issue #8700, "Design points": a parameter whose flat range lies in
// exactly one optimizer partition has that partition's rank as owner; one
// that straddles a boundary keeps AllReduce (-1); a group reduced over another
// communicator is excluded.  The device form is for executors that keep the
// parameter table in device memory (a graph-captured step, for instance).  One
// CTA walks the group in chunks of 1024 parameters: a warp-shuffle reduction
// gives the group's total T (and so the partition size ceil(T/S)), a
// warp-shuffle exclusive scan gives every parameter's flat start, and the
// owned parameters are counted with warp ballots.
#include "common.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int64_t warp_inclusive_scan(int64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += u;
    }
    return v;
}

__device__ __forceinline__ int64_t warp_sum(int64_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

__global__ void __launch_bounds__(kThreads) owner_map_kernel(int world, int n_params, const int64_t* __restrict__ numel,
                                                             int comm_size, const int32_t* __restrict__ comm_ranks,
                                                             int reduce_to_owner, int32_t* __restrict__ owner,
                                                             int32_t* __restrict__ holder_lo,
                                                             int32_t* __restrict__ holder_hi,
                                                             int32_t* __restrict__ counts) {
    __shared__ int64_t warp_part[kWarps];
    __shared__ int64_t s_total, s_carry;
    __shared__ int s_eligible, s_owned;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_eligible = comm_size == world;
        s_owned = 0;
        s_carry = 0;
    }
    __syncthreads();
    // eligibility: group rank i must be global rank i for every i
    for (int i = tid; comm_ranks && i < comm_size; i += kThreads)
        if (comm_ranks[i] != i) s_eligible = 0;
    // pass 1: T = sum of sizes
    int64_t acc = 0;
    for (int i = tid; i < n_params; i += kThreads) acc += numel[i];
    acc = warp_sum(acc);
    if (lane == 0) warp_part[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        int64_t v = lane < kWarps ? warp_part[lane] : 0;
        v = warp_sum(v);
        if (lane == 0) s_total = v;
    }
    __syncthreads();
    const int64_t T = s_total;
    const int64_t P = (T + comm_size - 1) / comm_size;
    const bool eligible = s_eligible != 0;
    // pass 2: exclusive scan of the sizes in chunks, then the map
    for (int base = 0; base < n_params; base += kThreads) {
        const int i = base + tid;
        const int64_t n = i < n_params ? numel[i] : 0;
        const int64_t incl = warp_inclusive_scan(n);
        if (lane == 31) warp_part[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int64_t w = lane < kWarps ? warp_part[lane] : 0;
            const int64_t wi = warp_inclusive_scan(w);
            if (lane < kWarps) warp_part[lane] = wi - w;  // exclusive prefix of the warp totals
        }
        __syncthreads();
        const int64_t s = s_carry + warp_part[warp] + (incl - n);  // flat start of parameter i
        bool owned = false;
        if (i < n_params) {
            int32_t o = -1, lo = -1, hi = -1;
            if (n > 0) {
                if (eligible) {
                    lo = (int32_t)(s / P);
                    hi = (int32_t)((s + n - 1) / P);
                    if (reduce_to_owner && lo == hi) o = lo;
                } else {
                    lo = 0;
                    hi = world - 1;
                }
            }
            owner[i] = o;
            holder_lo[i] = lo;
            holder_hi[i] = hi;
            owned = o >= 0;
        }
        const unsigned ball = __ballot_sync(0xffffffffu, owned);
        if (lane == 0 && ball) atomicAdd(&s_owned, __popc(ball));
        __syncthreads();
        if (tid == kThreads - 1) s_carry = s + n;  // the last thread's end is the next chunk's start
        __syncthreads();
    }
    if (tid == 0) {
        counts[0] = s_owned;
        counts[1] = n_params;
    }
}

}  // namespace

extern "C" int dpred_build_owner_map_device(int32_t world, int32_t n_params, const int64_t* numel, int32_t comm_size,
                                            const int32_t* comm_ranks, int32_t reduce_to_owner, int32_t* owner,
                                            int32_t* holder_lo, int32_t* holder_hi, int32_t* counts, void* stream) {
    if (world < 1 || world > DPRED_MAX_WORLD)
        return dpred::set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n_params < 0 || comm_size < 1) return dpred::set_error(DPRED_E_INVAL, "n_params < 0 or comm_size < 1");
    if (!counts || (n_params > 0 && (!numel || !owner || !holder_lo || !holder_hi)))
        return dpred::set_error(DPRED_E_INVAL, "null pointer");
    if (reinterpret_cast<uintptr_t>(numel) % 8 || reinterpret_cast<uintptr_t>(owner) % 4 ||
        reinterpret_cast<uintptr_t>(holder_lo) % 4 || reinterpret_cast<uintptr_t>(holder_hi) % 4 ||
        reinterpret_cast<uintptr_t>(counts) % 4 || reinterpret_cast<uintptr_t>(comm_ranks) % 4)
        return dpred::set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    owner_map_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        world, n_params, numel, comm_size, comm_ranks, reduce_to_owner, owner, holder_lo, holder_hi, counts);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "owner map kernel launch");
}
