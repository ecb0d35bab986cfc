// schedule.cu -- step-by-step AllGather schedules on one GPU.
//
// Page "AllGather" (tier6-model interconnect notes): "Ring AllGather" (N-1
// steps; each node forwards the chunk it received last step to its right
// neighbour), the bidirectional ring (eq. ag-bidir-ring, ceil((N-1)/2) steps,
// both directions at once) and "Recursive Doubling AllGather" (log2 N steps;
// in step j node i swaps everything it holds with node i xor 2^(j-1)).  The N
// node buffers are the N rows of one [N, N*S] array; row i, slot c holds a
// shard of S elements.  Each step is one launch of the plan-driven copy kernel
// that moves exactly the chunks the schedule sends in that step, so the
// buffers can be checked against the page's tables after every step and the
// per-step times fitted to the alpha-beta cost model.
#include <vector>

#include "common.cuh"

namespace {

int log2_exact(int n) {
    int k = 0;
    while ((1 << k) < n) ++k;
    return (1 << k) == n ? k : -1;
}

int steps_of(int schedule, int n) {
    switch (schedule) {
        case DPRED_SCHED_RING: return n - 1;
        case DPRED_SCHED_BIDIR_RING: return n / 2;
        case DPRED_SCHED_RECURSIVE_DOUBLING: return log2_exact(n);
        default: return -1;
    }
}

int check(int schedule, int n, int64_t shard, int dtype, const void* p) {
    if (n < 1 || n > DPRED_MAX_WORLD) return dpred::set_error(DPRED_E_INVAL, "n_nodes %d outside 1..%d", n, DPRED_MAX_WORLD);
    if (schedule < 0 || schedule > 2) return dpred::set_error(DPRED_E_INVAL, "unknown schedule %d", schedule);
    if (steps_of(schedule, n) < 0)
        return dpred::set_error(DPRED_E_INVAL, "recursive doubling needs a power-of-two node count, got %d", n);
    if (shard < 0) return dpred::set_error(DPRED_E_INVAL, "shard_elems < 0");
    if (dtype != DPRED_BF16 && dtype != DPRED_F32) return dpred::set_error(DPRED_E_INVAL, "bad dtype");
    if (shard > 0 && !p) return dpred::set_error(DPRED_E_INVAL, "null pointer");
    if (p && reinterpret_cast<uintptr_t>(p) % (dtype == DPRED_BF16 ? 2 : 4))
        return dpred::set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    return DPRED_OK;
}

}  // namespace

extern "C" {

int dpred_allgather_schedule_steps(int32_t schedule, int32_t n_nodes) {
    int rc = check(schedule, n_nodes, 0, DPRED_BF16, nullptr);
    return rc ? rc : steps_of(schedule, n_nodes);
}

int dpred_allgather_schedule_init(int32_t schedule, int32_t n_nodes, int64_t shard_elems, int32_t dtype,
                                  const void* in, void* bufs, void* stream) {
    int rc = check(schedule, n_nodes, shard_elems, dtype, bufs);
    if (rc == DPRED_OK) rc = check(schedule, n_nodes, shard_elems, dtype, in);
    if (rc) return rc;
    const int64_t cb = shard_elems * (dtype == DPRED_BF16 ? 2 : 4);  // chunk bytes
    std::vector<int64_t> t;
    for (int i = 0; i < n_nodes; ++i) {
        const int slot = schedule == DPRED_SCHED_RING ? 0 : i;  // ring lists start with the own chunk
        // source offsets are relative to `in`, destinations to `bufs`: copy through two plans
        t.insert(t.end(), {(int64_t)i * cb, ((int64_t)i * n_nodes + slot) * cb, cb});
    }
    return dpred::launch_copy_plan(static_cast<const char*>(in), static_cast<char*>(bufs), t, nullptr, 0,
                                   static_cast<cudaStream_t>(stream));
}

int dpred_allgather_schedule_step(int32_t schedule, int32_t n_nodes, int64_t shard_elems, int32_t dtype, void* bufs,
                                  int32_t step, void* stream) {
    int rc = check(schedule, n_nodes, shard_elems, dtype, bufs);
    if (rc) return rc;
    const int steps = steps_of(schedule, n_nodes);
    if (step < 1 || step > steps) return dpred::set_error(DPRED_E_INVAL, "step %d outside 1..%d", step, steps);
    const int N = n_nodes;
    const int64_t cb = shard_elems * (dtype == DPRED_BF16 ? 2 : 4);
    auto slot = [&](int node, int c) { return ((int64_t)node * N + c) * cb; };
    std::vector<int64_t> t;
    for (int i = 0; i < N; ++i) {
        if (schedule == DPRED_SCHED_RING) {
            // the chunk the left neighbour received last step (its slot step-1) lands in slot `step`
            t.insert(t.end(), {slot((i - 1 + N) % N, step - 1), slot(i, step), cb});
        } else if (schedule == DPRED_SCHED_BIDIR_RING) {
            const int left = ((i - step) % N + N) % N, right = (i + step) % N;
            t.insert(t.end(), {slot((i - 1 + N) % N, left), slot(i, left), cb});
            if (right != left) t.insert(t.end(), {slot((i + 1) % N, right), slot(i, right), cb});
        } else {
            const int d = 1 << (step - 1), partner = i ^ d, base = partner & ~(d - 1);
            t.insert(t.end(), {slot(partner, base), slot(i, base), (int64_t)d * cb});
        }
    }
    return dpred::launch_copy_plan(static_cast<const char*>(bufs), static_cast<char*>(bufs), t, nullptr, 0,
                                   static_cast<cudaStream_t>(stream));
}

}  // extern "C"
