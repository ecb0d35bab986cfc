// abi.cu -- the extern "C" entry points of libdpred: argument validation, the
// owner map and probe counters (host metadata), and the flush plan that the
// kernels execute.  Every entry point validates everything before enqueuing
// any device work and reports failures as DPRED_E_* codes, never by aborting.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace dpred {

__device__ int g_device_error;  // first device-side failure code, 0 when none

namespace {
int g_flush_path = PATH_AUTO;
}

// Tasks with no destination write nothing and are left out of the plan.
void build_plan(int world, int in_dt, const void* grads, int64_t ld, int out_dt, int pre_div,
                const std::vector<Dest>& tasks, BuiltPlan& out) {
    const int vec_elems = in_dt == DPRED_BF16 ? 8 : 4;
    const int isz = in_dt == DPRED_BF16 ? 2 : 4, osz = out_dt == DPRED_BF16 ? 2 : 4;
    const size_t out_align = std::min<size_t>(16, (size_t)vec_elems * osz);
    const bool rows_vec = reinterpret_cast<uintptr_t>(grads) % 16 == 0 && (ld * isz) % 16 == 0;
    out.tasks.clear();
    out.pool.clear();
    out.realign = false;
    out.write_heavy = false;
    int64_t read_bytes = 0, write_bytes = 0;
    out.tasks.reserve(tasks.size());
    int64_t units = 0;
    const int unit_vec = kUnitVec * flush_batch(world, in_dt == DPRED_BF16);
    for (const Dest& d : tasks) {
        if (d.numel == 0 || d.ptrs.empty()) continue;
        TaskDesc t{};
        t.src_off = d.src_off;
        t.numel = d.numel;
        t.dst_begin = (int32_t)out.pool.size();
        t.ndst = (int16_t)d.ptrs.size();
        int64_t head = (vec_elems - d.src_off % vec_elems) % vec_elems;
        if (head > d.numel) head = d.numel;
        bool vec = rows_vec;
        for (void* p : d.ptrs)
            if ((reinterpret_cast<uintptr_t>(p) + (uintptr_t)head * osz) % out_align != 0) vec = false;
        int mode = vec ? 1 : 0;
        if (!vec && rows_vec && in_dt == out_dt && (d.numel - head) / vec_elems >= 2) {
            // Same element type, destinations shifted against the source grid:
            // the realigned vector path when every destination has the same shift.
            int sigma = -1;
            for (void* p : d.ptrs) {
                const int64_t de = (int64_t)(reinterpret_cast<uintptr_t>(p) / (uintptr_t)osz);
                const int64_t a = (vec_elems - de % vec_elems) % vec_elems;  // first 16-byte aligned element
                const int sg = (int)(((head - a) % vec_elems + vec_elems) % vec_elems);
                if (sigma < 0) {
                    sigma = sg;
                } else if (sg != sigma) {
                    sigma = 0;
                    break;
                }
            }
            if (sigma > 0) mode = 1 + sigma;
        }
        t.vec = (uint8_t)mode;
        t.head = mode ? (uint8_t)head : 0;
        if (mode >= 2) out.realign = true;
        t.unit_begin = units;
        units += flush_task_units(t, vec_elems, unit_vec);
        out.pool.insert(out.pool.end(), d.ptrs.begin(), d.ptrs.end());
        out.tasks.push_back(t);
        read_bytes += (int64_t)world * d.numel * isz;
        write_bytes += (int64_t)d.ptrs.size() * d.numel * osz;
    }
    out.write_heavy = 2 * write_bytes >= read_bytes && read_bytes > 0;
    out.h = FlushHeader{};
    out.h.grads = grads;
    out.h.ld = ld;
    out.h.total_units = units;
    out.h.world = world;
    out.h.n_tasks = (int32_t)out.tasks.size();
    out.h.pdiv = (pre_div && world > 1) ? (((world & (world - 1)) == 0) ? PDIV_POW2 : PDIV_DIV) : PDIV_NONE;
    out.h.wf = (float)world;
    out.h.inv_w = 1.0f / (float)world;
    out.h.unit_vec = unit_vec;
    prediv_split(world, &out.h.c_hi, &out.h.c_lo);
    out.in_dt = in_dt;
    out.out_dt = out_dt;
}

void prediv_split(int world, float* c_hi, float* c_lo) {
    const double inv = 1.0 / (double)world;
    int e = 0;
    const double m = std::frexp(inv, &e);  // inv = m * 2^e, m in [0.5, 1)
    const double hi = std::ldexp(std::floor(std::ldexp(m, 16)), e - 16);
    *c_hi = (float)hi;                     // 16 significant bits: exact
    *c_lo = (float)(inv - hi);             // the difference is exact in double
}

int launch_plan(const BuiltPlan& p, void* workspace, size_t workspace_bytes, cudaStream_t s, bool pdl) {
    if (p.tasks.empty()) return DPRED_OK;
    FlushLaunch L{};
    L.h = p.h;
    L.h.err = device_error_word();
    L.in_dt = p.in_dt;
    L.out_dt = p.out_dt;
    L.tasks = p.tasks.data();
    L.dst = p.pool.data();
    L.n_dst = (int)p.pool.size();
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.realign = p.realign;
    L.ldg_only = p.ldg_only;
    L.pdl = pdl;
    L.write_heavy = p.write_heavy;
    return p.in_dt == DPRED_BF16 ? launch_flush_bf16_in(L, s) : launch_flush_f32_in(L, s);
}

int flush_path() { return g_flush_path; }

int refuse_capture_of_upload(cudaStream_t s, const char* what) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_error(e, "stream capture query");
    if (cs != cudaStreamCaptureStatusNone)
        return set_error(DPRED_E_INVAL,
                         "%s does not fit inside the launch and is uploaded from host memory, which a CUDA graph "
                         "cannot capture; capture only plans with no workspace",
                         what);
    return DPRED_OK;
}

namespace {
thread_local std::string t_last_error;

int elem_size(int dt) { return dt == DPRED_BF16 ? 2 : 4; }
bool dtype_ok(int dt) { return dt == DPRED_BF16 || dt == DPRED_F32; }
bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }
bool pow2(int w) { return w > 0 && (w & (w - 1)) == 0; }

// Turn per-task destination lists into a kernel plan and launch it.
int run_plan(int world, int in_dt, const void* grads, int64_t ld, int out_dt, int pre_div,
             const std::vector<Dest>& tasks, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    BuiltPlan p;
    build_plan(world, in_dt, grads, ld, out_dt, pre_div, tasks, p);
    return launch_plan(p, workspace, workspace_bytes, s);
}

}  // namespace

int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_error(cudaError_t e, const char* what) {
    return set_error(DPRED_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

int resident_ctas(const void* kernel, int threads) {
    struct Entry {
        const void* kernel;
        int threads, dev, occ;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
        if (e.kernel == kernel && e.threads == threads && e.dev == dev) return e.occ;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, 0) != cudaSuccess || occ < 1) occ = 1;
    cache.push_back(Entry{kernel, threads, dev, occ});
    return occ;
}

int* device_error_word() {
    static int* cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (cached[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<int*>(p);
    }
    return cached[dev];
}

}  // namespace dpred

using namespace dpred;

extern "C" {

const char* dpred_last_error(void) { return t_last_error.c_str(); }

const char* dpred_version(void) { return "dpred 0.1 (sm_103a)"; }

int dpred_checked_build(void) {
#if defined(DPRED_CHECKED) && DPRED_CHECKED
    return 1;
#else
    return 0;
#endif
}

int dpred_build_owner_map(int32_t world, int32_t rank, const dpred_group* groups, int32_t n_groups,
                          int32_t reduce_to_owner, int32_t* owner, int32_t* holder_lo, int32_t* holder_hi,
                          int32_t* n_owned, int32_t* n_total) {
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (rank < 0 || rank >= world) return set_error(DPRED_E_INVAL, "rank %d outside 0..%d", rank, world - 1);
    if (n_groups < 0 || (n_groups > 0 && groups == nullptr))
        return set_error(DPRED_E_INVAL, "bad group list");
    if (!n_owned || !n_total) return set_error(DPRED_E_INVAL, "null count output");
    int64_t n_all = 0;
    for (int g = 0; g < n_groups; ++g) {
        const dpred_group& G = groups[g];
        if (G.comm_size < 1 || G.n_params < 0 || (G.n_params > 0 && G.numel == nullptr))
            return set_error(DPRED_E_INVAL, "group %d: bad comm_size / n_params / numel", g);
        for (int p = 0; p < G.n_params; ++p)
            if (G.numel[p] < 0) return set_error(DPRED_E_INVAL, "group %d param %d: negative size", g, p);
        n_all += G.n_params;
    }
    if (n_all > 0 && (!owner || !holder_lo || !holder_hi)) return set_error(DPRED_E_INVAL, "null map output");
    int32_t owned = 0, total = 0;
    int64_t out = 0;
    for (int g = 0; g < n_groups; ++g) {
        const dpred_group& G = groups[g];
        bool eligible = G.comm_size == world;
        for (int i = 0; eligible && G.comm_ranks && i < G.comm_size; ++i) eligible = G.comm_ranks[i] == i;
        int64_t T = 0;
        for (int p = 0; p < G.n_params; ++p) T += G.numel[p];
        const int64_t P = (T + G.comm_size - 1) / G.comm_size;
        int64_t s = 0;
        for (int p = 0; p < G.n_params; ++p, ++out) {
            const int64_t n = G.numel[p];
            if (n == 0) {
                owner[out] = holder_lo[out] = holder_hi[out] = -1;
            } else if (!eligible) {
                owner[out] = -1;
                holder_lo[out] = 0;
                holder_hi[out] = world - 1;
            } else {
                const int32_t lo = (int32_t)(s / P), hi = (int32_t)((s + n - 1) / P);
                holder_lo[out] = lo;
                holder_hi[out] = hi;
                owner[out] = (reduce_to_owner && lo == hi) ? lo : -1;
            }
            owned += owner[out] >= 0;
            ++total;
            s += n;
        }
    }
    *n_owned = owned;
    *n_total = total;
    return DPRED_OK;
}

uint64_t dpred_owner_map_digest(int32_t n_params, const int32_t* owner, const int32_t* holder_lo,
                                const int32_t* holder_hi) {
    // FNV-1a (64-bit) over the parameter count and the three arrays, little-endian
    uint64_t h = 0xcbf29ce484222325ull;
    auto mix = [&h](uint32_t v) {
        for (int b = 0; b < 4; ++b) {
            h ^= (v >> (8 * b)) & 0xffu;
            h *= 0x100000001b3ull;
        }
    };
    mix((uint32_t)n_params);
    const int32_t* arrays[3] = {owner, holder_lo, holder_hi};
    for (const int32_t* a : arrays)
        for (int32_t i = 0; a && i < n_params; ++i) mix((uint32_t)a[i]);
    return h;
}

static int validate_tasks(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                          int32_t n_params, int64_t ld, bool check_ld) {
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n_tasks < 0 || (n_tasks > 0 && tasks == nullptr)) return set_error(DPRED_E_INVAL, "bad task list");
    if (owner && n_params < 0) return set_error(DPRED_E_INVAL, "n_params < 0");
    for (int t = 0; t < n_tasks; ++t) {
        const dpred_task& k = tasks[t];
        if (k.reserved != 0) return set_error(DPRED_E_INVAL, "task %d: reserved field must be 0", t);
        if (k.offset < 0 || k.numel < 0) return set_error(DPRED_E_INVAL, "task %d: negative offset or size", t);
        if (check_ld && k.offset + k.numel > ld)
            return set_error(DPRED_E_SIZE, "task %d: [%lld, %lld) outside the row of %lld elements", t,
                             (long long)k.offset, (long long)(k.offset + k.numel), (long long)ld);
        if (owner) {
            if (k.param_id < 0 || k.param_id >= n_params)
                return set_error(DPRED_E_INVAL, "task %d: param_id %d outside 0..%d", t, k.param_id, n_params - 1);
            if (owner[k.param_id] < -1 || owner[k.param_id] >= world)
                return set_error(DPRED_E_INVAL, "owner of param %d is %d, not a rank", k.param_id, owner[k.param_id]);
        }
    }
    return DPRED_OK;
}

static int root_of(const dpred_task& k, const int32_t* owner, int32_t reduce_to_owner) {
    return (reduce_to_owner && owner && owner[k.param_id] >= 0) ? owner[k.param_id] : -1;
}

static void fill_probe(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                       void* const* dst, int32_t reduce_to_owner, dpred_probe* probe) {
    probe->tasks = n_tasks;
    probe->reduced_elems = probe->owner_tasks = probe->owner_elems = 0;
    for (int r = 0; r < DPRED_MAX_WORLD; ++r) probe->kept_elems[r] = 0;
    for (int t = 0; t < n_tasks; ++t) {
        const int root = root_of(tasks[t], owner, reduce_to_owner);
        probe->reduced_elems += tasks[t].numel;
        if (root >= 0) {
            probe->owner_tasks += 1;
            probe->owner_elems += tasks[t].numel;
        }
        for (int r = 0; r < world; ++r) {
            bool kept = dst ? dst[(int64_t)r * n_tasks + t] != nullptr : (root < 0 || root == r);
            if (kept) probe->kept_elems[r] += tasks[t].numel;
        }
    }
}

int dpred_flush_probe(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                      int32_t n_params, void* const* dst, int32_t reduce_to_owner, dpred_probe* probe) {
    int rc = validate_tasks(world, tasks, n_tasks, owner, n_params, 0, false);
    if (rc) return rc;
    if (!probe) return set_error(DPRED_E_INVAL, "null probe");
    fill_probe(world, tasks, n_tasks, owner, dst, reduce_to_owner, probe);
    return DPRED_OK;
}

int dpred_probe_format(const dpred_probe* probe, int32_t world, int32_t rank, int32_t dtype, int32_t pre_div,
                       char* buf, size_t buf_bytes) {
    if (!probe || !buf) return set_error(DPRED_E_INVAL, "null probe or buffer");
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (rank < 0 || rank >= world) return set_error(DPRED_E_INVAL, "rank %d outside 0..%d", rank, world - 1);
    if (!dtype_ok(dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    const long long red = probe->reduced_elems, kept = probe->kept_elems[rank];
    const double discarded = red ? 100.0 * (double)(red - kept) / (double)red : 0.0;
    const double owner_pct = red ? 100.0 * (double)probe->owner_elems / (double)red : 0.0;
    const int n = std::snprintf(buf, buf_bytes,
                                "[dc-probe][r%d] flushReduceBucket #%lld dtype=%s tasks=%lld reduced_elems=%lld "
                                "kept_elems=%lld discarded=%.1f%% pre_div=%d owner_tasks=%lld owner_elems=%lld (%.1f%%)",
                                rank, (long long)probe->flush_index, dtype == DPRED_BF16 ? "BFloat16" : "Float",
                                (long long)probe->tasks, red, kept, discarded, pre_div ? 1 : 0,
                                (long long)probe->owner_tasks, (long long)probe->owner_elems, owner_pct);
    if (n < 0) return set_error(DPRED_E_INVAL, "probe line formatting failed");
    if ((size_t)n >= buf_bytes)
        return set_error(DPRED_E_SIZE, "probe line needs %d bytes plus the terminator, buffer holds %zu", n, buf_bytes);
    return DPRED_OK;
}

size_t dpred_flush_workspace_bytes(int32_t world, int32_t n_tasks) {
    if (world < 1 || n_tasks < 0) return 0;
    const int64_t dsts = (int64_t)world * n_tasks;
    if (n_tasks <= kInlineTasks && dsts <= kInlineDst) return 0;
    return sizeof(TaskDesc) * (size_t)n_tasks + (((size_t)dsts * sizeof(void*) + 15) & ~(size_t)15);
}

}  // extern "C"

namespace {

// The per-call plan cache of dpred_flush_bucket.  A training step flushes the
// same buckets with the same tables every step; validating them, computing
// the probe counters and building the launch plan again each time is pure
// host overhead.  Each entry keeps the exact inputs a plan was built from --
// scalars, the task table, the owner of every task's parameter and the
// destination table -- and a call whose inputs compare equal byte for byte
// reuses the entry's validated plan and counters.  The plan depends on the
// destination pointers' values only (never on the memory behind them), so a
// cached plan is as valid as a rebuilt one.  One cache per thread, no locks.
struct CachedFlush {
    int32_t world = 0, in_dt = 0, out_dt = 0, pre_div = 0, rto = 0, n_tasks = 0, n_params = 0;
    const void* grads = nullptr;
    int64_t ld = 0;
    bool has_owner = false, has_dst = false;
    bool checked_ok = false;  // the checked-mode ownership test passed for these inputs
    std::vector<dpred_task> tasks;
    std::vector<int32_t> owner_of_task;  // owner[param_id] of every task (when owner != NULL)
    std::vector<void*> dst;              // [world * n_tasks] when dst != NULL
    dpred_probe probe{};                 // counters; flush_index comes from each call
    BuiltPlan plan;
    uint64_t last_use = 0;
};
constexpr size_t kFlushCacheEntries = 16;
thread_local std::vector<CachedFlush> t_flush_cache;
thread_local uint64_t t_flush_clock = 0;
thread_local std::vector<Dest> t_dests;  // plan scratch reused across calls (no allocation per task)

bool same_inputs(const CachedFlush& c, int32_t world, int32_t in_dtype, const void* grads, int64_t ld,
                 const dpred_task* tasks, int32_t n_tasks, const int32_t* owner, int32_t n_params, int32_t out_dtype,
                 void* const* dst, int32_t pre_div, int32_t reduce_to_owner) {
    if (c.world != world || c.in_dt != in_dtype || c.out_dt != out_dtype || c.grads != grads || c.ld != ld ||
        c.n_tasks != n_tasks || c.pre_div != (pre_div != 0) || c.rto != (reduce_to_owner != 0) ||
        c.has_owner != (owner != nullptr) || c.has_dst != (dst != nullptr) || (owner && c.n_params != n_params))
        return false;
    if (n_tasks && std::memcmp(c.tasks.data(), tasks, sizeof(dpred_task) * (size_t)n_tasks) != 0) return false;
    // the task table equals a validated one, so every param_id is inside owner[0, n_params)
    if (owner)
        for (int32_t t = 0; t < n_tasks; ++t)
            if (owner[tasks[t].param_id] != c.owner_of_task[t]) return false;
    if (dst && n_tasks && std::memcmp(c.dst.data(), dst, sizeof(void*) * (size_t)world * n_tasks) != 0) return false;
    return true;
}

int check_ownership(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                    void* const* dst, int32_t reduce_to_owner) {
    for (int t = 0; t < n_tasks; ++t) {
        const int root = root_of(tasks[t], owner, reduce_to_owner);
        if (root < 0) continue;
        for (int r = 0; r < world; ++r)
            if (r != root && dst[(int64_t)r * n_tasks + t] != nullptr)
                return set_error(DPRED_E_MISMATCH,
                                 "task %d (param %d) is owned by rank %d but rank %d has a non-empty buffer", t,
                                 tasks[t].param_id, root, r);
    }
    return DPRED_OK;
}

}  // namespace

extern "C" {

int dpred_flush_bucket(int32_t world, int32_t in_dtype, void* grads, int64_t ld, const dpred_task* tasks,
                       int32_t n_tasks, const int32_t* owner, int32_t n_params, int32_t out_dtype, void* const* dst,
                       int32_t pre_div, int32_t reduce_to_owner, int32_t flags, dpred_probe* probe,
                       void* workspace, size_t workspace_bytes, void* stream) {
    if (flags & ~(DPRED_FLUSH_CHECKED | DPRED_FLUSH_OVERLAP))
        return set_error(DPRED_E_INVAL, "unknown flush flags 0x%x", (unsigned)flags);
    const bool checked = (flags & DPRED_FLUSH_CHECKED) != 0;
    const bool overlap = (flags & DPRED_FLUSH_OVERLAP) != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a repeated call: the same inputs were validated and planned before
    for (CachedFlush& c : t_flush_cache) {
        if (!same_inputs(c, world, in_dtype, grads, ld, tasks, n_tasks, owner, n_params, out_dtype, dst, pre_div,
                         reduce_to_owner))
            continue;
        if (checked && dst && !c.checked_ok) {
            int rc = check_ownership(world, tasks, n_tasks, owner, dst, reduce_to_owner);
            if (rc) return rc;
            c.checked_ok = true;
        }
        c.last_use = ++t_flush_clock;
        if (probe) {
            const int64_t idx = probe->flush_index;
            *probe = c.probe;
            probe->flush_index = idx;
        }
        return launch_plan(c.plan, workspace, workspace_bytes, s, overlap);
    }

    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (ld < 0) return set_error(DPRED_E_INVAL, "ld < 0");
    int rc = validate_tasks(world, tasks, n_tasks, owner, n_params, ld, true);
    if (rc) return rc;
    const int isz = elem_size(in_dtype), osz = elem_size(out_dtype);
    bool any = false;
    for (int t = 0; t < n_tasks; ++t) any |= tasks[t].numel > 0;
    if (any && grads == nullptr) return set_error(DPRED_E_INVAL, "null grads");
    if (grads && !aligned(grads, isz)) return set_error(DPRED_E_ALIGN, "grads not aligned to its element size");
    if (dst == nullptr) {
        if (out_dtype != in_dtype) return set_error(DPRED_E_INVAL, "in-place flush needs out_dtype == in_dtype");
        std::vector<std::pair<int64_t, int64_t>> r;
        for (int t = 0; t < n_tasks; ++t)
            if (tasks[t].numel > 0) r.emplace_back(tasks[t].offset, tasks[t].offset + tasks[t].numel);
        std::sort(r.begin(), r.end());
        for (size_t i = 1; i < r.size(); ++i)
            if (r[i].first < r[i - 1].second) return set_error(DPRED_E_SIZE, "in-place tasks overlap");
    } else {
        for (int64_t i = 0; i < (int64_t)world * n_tasks; ++i)
            if (dst[i] && !aligned(dst[i], osz))
                return set_error(DPRED_E_ALIGN, "destination %lld not aligned to its element size", (long long)i);
    }
    if (checked && dst) {
        rc = check_ownership(world, tasks, n_tasks, owner, dst, reduce_to_owner);
        if (rc) return rc;
    }

    // a new entry (the least recently used one makes room)
    CachedFlush* c;
    if (t_flush_cache.size() < kFlushCacheEntries) {
        t_flush_cache.emplace_back();
        c = &t_flush_cache.back();
    } else {
        c = &*std::min_element(t_flush_cache.begin(), t_flush_cache.end(),
                               [](const CachedFlush& a, const CachedFlush& b) { return a.last_use < b.last_use; });
    }
    c->world = world;
    c->in_dt = in_dtype;
    c->out_dt = out_dtype;
    c->grads = grads;
    c->ld = ld;
    c->n_tasks = n_tasks;
    c->n_params = n_params;
    c->pre_div = pre_div != 0;
    c->rto = reduce_to_owner != 0;
    c->has_owner = owner != nullptr;
    c->has_dst = dst != nullptr;
    c->checked_ok = checked && dst;
    c->tasks.assign(tasks, tasks + n_tasks);
    c->owner_of_task.clear();
    if (owner)
        for (int t = 0; t < n_tasks; ++t) c->owner_of_task.push_back(owner[tasks[t].param_id]);
    c->dst.clear();
    if (dst) c->dst.assign(dst, dst + (int64_t)world * n_tasks);
    fill_probe(world, tasks, n_tasks, owner, dst, reduce_to_owner, &c->probe);
    c->last_use = ++t_flush_clock;

    std::vector<Dest>& plan = t_dests;
    plan.resize((size_t)n_tasks);
    for (int t = 0; t < n_tasks; ++t) {
        const int root = root_of(tasks[t], owner, reduce_to_owner);
        Dest& d = plan[t];
        d.src_off = tasks[t].offset;
        d.numel = tasks[t].numel;
        d.ptrs.clear();
        for (int r = 0; r < world; ++r) {
            if (root >= 0 && r != root) continue;  // not delivered: untouched
            void* p = dst ? dst[(int64_t)r * n_tasks + t]
                          : static_cast<char*>(grads) + ((int64_t)r * ld + tasks[t].offset) * isz;
            if (p) d.ptrs.push_back(p);  // empty buffer: skipped in the copy-out
        }
    }
    build_plan(world, in_dtype, grads, ld, out_dtype, pre_div, plan, c->plan);
    if (probe) {
        const int64_t idx = probe->flush_index;
        *probe = c->probe;
        probe->flush_index = idx;
    }
    return launch_plan(c->plan, workspace, workspace_bytes, s, overlap);
}

int dpred_accumulate_microbatch(int32_t world, int64_t n, float* acc, int32_t g_dtype, const void* g,
                                int32_t first, int32_t finalize, float scale, float* total, void* stream) {
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n < 0) return set_error(DPRED_E_INVAL, "n < 0");
    if (!dtype_ok(g_dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (n > 0 && (!acc || !g || (finalize && !total))) return set_error(DPRED_E_INVAL, "null pointer");
    if ((acc && !aligned(acc, 4)) || (g && !aligned(g, elem_size(g_dtype))) || (total && !aligned(total, 4)))
        return set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    return launch_accumulate(world, n, acc, g_dtype, g, first, finalize, scale, total,
                             static_cast<cudaStream_t>(stream));
}

// Pieces of a bucket cut at partition boundaries: {task, rank, flat lo, flat hi}.
struct PartPiece {
    int task, rank;
    int64_t lo, hi;
};

static int partition_pieces(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int64_t* flat_offset,
                            int32_t n_params, int64_t part_size, std::vector<PartPiece>& out) {
    if (!flat_offset && n_tasks > 0) return set_error(DPRED_E_INVAL, "null flat_offset");
    if (part_size < 1) return set_error(DPRED_E_INVAL, "part_size < 1");
    for (int t = 0; t < n_tasks; ++t) {
        const dpred_task& k = tasks[t];
        if (k.param_id < 0 || k.param_id >= n_params)
            return set_error(DPRED_E_INVAL, "task %d: param_id %d outside 0..%d", t, k.param_id, n_params - 1);
        if (k.numel == 0) continue;
        const int64_t s = flat_offset[k.param_id], e = s + k.numel;
        if (s < 0 || (e - 1) / part_size >= world)
            return set_error(DPRED_E_SIZE, "task %d: flat range [%lld, %lld) outside %d partitions of %lld", t,
                             (long long)s, (long long)e, world, (long long)part_size);
        for (int64_t r = s / part_size; r <= (e - 1) / part_size; ++r)
            out.push_back(PartPiece{t, (int)r, std::max(s, r * part_size), std::min(e, (r + 1) * part_size)});
    }
    std::vector<std::pair<int64_t, int64_t>> ranges;
    for (const PartPiece& p : out) ranges.emplace_back(p.lo, p.hi);
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second) return set_error(DPRED_E_SIZE, "tasks overlap in the flat space");
    return DPRED_OK;
}

}  // extern "C"

namespace dpred {

// The plan and probe of one partitioned flush: validation, the pieces of every
// task cut at the partition boundaries, and one destination per piece inside
// its rank's partition buffer.  Shared by dpred_flush_bucket_partitioned and
// the partitioned executor.
int partitioned_plan(int32_t world, int32_t in_dtype, int32_t out_dtype, const void* grads, int64_t ld,
                     const dpred_task* tasks, int32_t n_tasks, const int64_t* flat_offset, int32_t n_params,
                     int64_t part_size, void* const* part_dst, std::vector<Dest>& plan, dpred_probe* probe) {
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (ld < 0) return set_error(DPRED_E_INVAL, "ld < 0");
    int rc = validate_tasks(world, tasks, n_tasks, nullptr, 0, ld, true);
    if (rc) return rc;
    if (n_tasks > 0 && !part_dst) return set_error(DPRED_E_INVAL, "null part_dst table");
    const int isz = elem_size(in_dtype), osz = elem_size(out_dtype);
    bool any = false;
    for (int t = 0; t < n_tasks; ++t) any |= tasks[t].numel > 0;
    if (any && !grads) return set_error(DPRED_E_INVAL, "null grads");
    if (grads && !aligned(grads, isz)) return set_error(DPRED_E_ALIGN, "grads not aligned to its element size");
    for (int r = 0; r < world && part_dst; ++r)
        if (part_dst[r] && !aligned(part_dst[r], osz)) return set_error(DPRED_E_ALIGN, "partition %d misaligned", r);
    std::vector<PartPiece> pieces;
    rc = partition_pieces(world, tasks, n_tasks, flat_offset, n_params, part_size, pieces);
    if (rc) return rc;
    if (probe) {
        probe->tasks = n_tasks;
        probe->reduced_elems = probe->owner_tasks = probe->owner_elems = 0;
        for (int r = 0; r < DPRED_MAX_WORLD; ++r) probe->kept_elems[r] = 0;
        for (int t = 0; t < n_tasks; ++t) {
            probe->reduced_elems += tasks[t].numel;
            if (tasks[t].numel == 0) continue;
            const int64_t s = flat_offset[tasks[t].param_id];
            if (s / part_size == (s + tasks[t].numel - 1) / part_size) {
                probe->owner_tasks += 1;
                probe->owner_elems += tasks[t].numel;
            }
        }
        for (const PartPiece& p : pieces)
            if (part_dst[p.rank]) probe->kept_elems[p.rank] += p.hi - p.lo;
    }
    plan.clear();
    plan.reserve(pieces.size());
    for (const PartPiece& p : pieces) {
        if (!part_dst[p.rank]) continue;
        Dest d;
        d.src_off = tasks[p.task].offset + (p.lo - flat_offset[tasks[p.task].param_id]);
        d.numel = p.hi - p.lo;
        d.ptrs.push_back(static_cast<char*>(part_dst[p.rank]) + (p.lo - p.rank * part_size) * osz);
        plan.push_back(std::move(d));
    }
    return DPRED_OK;
}

}  // namespace dpred

extern "C" {

int dpred_flush_bucket_partitioned(int32_t world, int32_t in_dtype, const void* grads, int64_t ld,
                                   const dpred_task* tasks, int32_t n_tasks, const int64_t* flat_offset,
                                   int32_t n_params, int64_t part_size, int32_t out_dtype, void* const* part_dst,
                                   int32_t pre_div, dpred_probe* probe, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    std::vector<Dest> plan;
    int rc = partitioned_plan(world, in_dtype, out_dtype, grads, ld, tasks, n_tasks, flat_offset, n_params, part_size,
                              part_dst, plan, probe);
    if (rc) return rc;
    return run_plan(world, in_dtype, grads, ld, out_dtype, pre_div, plan, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
}

size_t dpred_bucket_relayout_workspace_bytes(int32_t world, int32_t n_tasks) {
    if (world < 1 || n_tasks < 0) return 0;
    return relayout_workspace_bytes((int64_t)world * ((int64_t)n_tasks + world - 1));
}

int dpred_bucket_relayout(int32_t world, int32_t dtype, const void* grads, int64_t ld, const dpred_task* tasks,
                          int32_t n_tasks, const int64_t* flat_offset, int32_t n_params, int64_t part_size, int64_t seg,
                          void* out, int64_t out_ld, int64_t* seg_used, void* workspace, size_t workspace_bytes,
                          void* stream) {
    if (!dtype_ok(dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (ld < 0 || seg < 0 || out_ld < (int64_t)world * seg) return set_error(DPRED_E_INVAL, "bad ld / seg / out_ld");
    if (!seg_used) return set_error(DPRED_E_INVAL, "null seg_used");
    int rc = validate_tasks(world, tasks, n_tasks, nullptr, 0, ld, true);
    if (rc) return rc;
    const int esz = elem_size(dtype);
    if ((grads && !aligned(grads, esz)) || (out && !aligned(out, esz)))
        return set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    std::vector<PartPiece> pieces;
    rc = partition_pieces(world, tasks, n_tasks, flat_offset, n_params, part_size, pieces);
    if (rc) return rc;
    std::vector<int64_t> first(world, -1);
    for (int r = 0; r < world; ++r) seg_used[r] = 0;
    for (const PartPiece& p : pieces) {
        if (first[p.rank] < 0 || p.lo < first[p.rank]) first[p.rank] = p.lo;
        seg_used[p.rank] += p.hi - p.lo;
    }
    for (int r = 0; r < world; ++r)
        if (seg_used[r] > seg) return set_error(DPRED_E_SIZE, "rank %d needs %lld elements, seg is %lld", r,
                                                (long long)seg_used[r], (long long)seg);
    for (const PartPiece& p : pieces)
        if (p.hi - first[p.rank] > seg_used[p.rank])
            return set_error(DPRED_E_INVAL, "the bucket's elements in partition %d are not one contiguous flat run", p.rank);
    if (!pieces.empty() && (!grads || !out)) return set_error(DPRED_E_INVAL, "null pointer");
    std::vector<int64_t> triples;
    triples.reserve(pieces.size() * world * 3);
    for (int q = 0; q < world; ++q)
        for (const PartPiece& p : pieces) {
            const dpred_task& k = tasks[p.task];
            triples.push_back(((int64_t)q * ld + k.offset + (p.lo - flat_offset[k.param_id])) * esz);
            triples.push_back(((int64_t)q * out_ld + (int64_t)p.rank * seg + (p.lo - first[p.rank])) * esz);
            triples.push_back((p.hi - p.lo) * esz);
        }
    return launch_copy_plan(static_cast<const char*>(grads), static_cast<char*>(out), triples, workspace,
                            workspace_bytes, static_cast<cudaStream_t>(stream));
}

static int check_acc_args(int32_t world, int64_t n, const float* acc, const float* total) {
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n < 0) return set_error(DPRED_E_INVAL, "n < 0");
    if (n > 0 && (!acc || !total)) return set_error(DPRED_E_INVAL, "null pointer");
    if ((acc && !aligned(acc, 4)) || (total && !aligned(total, 4)))
        return set_error(DPRED_E_ALIGN, "pointer not aligned to 4 bytes");
    return DPRED_OK;
}

int dpred_accumulator_save(int32_t world, int64_t n, const float* acc, float* total, void* stream) {
    int rc = check_acc_args(world, n, acc, total);
    return rc ? rc : launch_accumulator_save(world, n, acc, total, static_cast<cudaStream_t>(stream));
}

int dpred_accumulator_restore(int32_t world, int64_t n, float* acc, const float* total, void* stream) {
    int rc = check_acc_args(world, n, acc, total);
    return rc ? rc : launch_accumulator_restore(world, n, acc, total, static_cast<cudaStream_t>(stream));
}

int dpred_reduce_scatter(int32_t n_nodes, int64_t m_elems, int32_t in_dtype, const void* in, int32_t out_dtype,
                         void* out, int32_t pre_div, void* stream) {
    if (n_nodes < 1 || n_nodes > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "n_nodes %d outside 1..%d", n_nodes, DPRED_MAX_WORLD);
    if (m_elems < 0) return set_error(DPRED_E_INVAL, "m_elems < 0");
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (m_elems % n_nodes != 0) return set_error(DPRED_E_SIZE, "M = %lld is not a multiple of N = %d", (long long)m_elems, n_nodes);
    if (m_elems > 0 && (!in || !out)) return set_error(DPRED_E_INVAL, "null pointer");
    if ((in && !aligned(in, elem_size(in_dtype))) || (out && !aligned(out, elem_size(out_dtype))))
        return set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    const int64_t S = m_elems / n_nodes;
    std::vector<Dest> plan(n_nodes);
    for (int i = 0; i < n_nodes; ++i) {
        plan[i].src_off = (int64_t)i * S;
        plan[i].numel = S;
        plan[i].ptrs.push_back(static_cast<char*>(out) + (int64_t)i * S * elem_size(out_dtype));
    }
    return run_plan(n_nodes, in_dtype, in, m_elems, out_dtype, pre_div, plan, nullptr, 0,
                    static_cast<cudaStream_t>(stream));
}

int dpred_allgather(int32_t n_nodes, int64_t shard_elems, int32_t dtype, const void* in, void* out, int32_t order,
                    void* stream) {
    if (n_nodes < 1 || n_nodes > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "n_nodes %d outside 1..%d", n_nodes, DPRED_MAX_WORLD);
    if (shard_elems < 0) return set_error(DPRED_E_INVAL, "shard_elems < 0");
    if (!dtype_ok(dtype)) return set_error(DPRED_E_INVAL, "bad dtype");
    if (order != 0 && order != 1) return set_error(DPRED_E_INVAL, "order must be 0 (canonical) or 1 (ring)");
    if (shard_elems > 0 && (!in || !out)) return set_error(DPRED_E_INVAL, "null pointer");
    const int esz = elem_size(dtype);
    if ((in && !aligned(in, esz)) || (out && !aligned(out, esz)))
        return set_error(DPRED_E_ALIGN, "pointer not aligned to its element size");
    return launch_allgather(n_nodes, shard_elems, esz, in, out, order, static_cast<cudaStream_t>(stream));
}

int dpred_set_flush_path(int32_t path) {
    if (path != PATH_AUTO && path != PATH_LDG && path != PATH_TMA)
        return set_error(DPRED_E_INVAL, "flush path %d: 0 (auto), 1 (LDG) or 2 (TMA)", path);
    int prev = g_flush_path;
    g_flush_path = path;
    return prev;
}

int dpred_set_allgather_form(int32_t form) {
    const int prev = set_allgather_form(form);
    if (prev < 0)
        return set_error(DPRED_E_INVAL, "allgather form %d: 0 (auto), 1 (register), 2 (TMA, one issuer), "
                                        "3 (TMA, four issuers) or 4 (TMA load, warp stores)", form);
    return prev;
}

int dpred_device_status(int32_t* code, int32_t clear) {
    if (!code) return set_error(DPRED_E_INVAL, "null code");
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_error(e, "reading the device error word");
    if (clear) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_error(e, "clearing the device error word");
    }
    return DPRED_OK;
}

}  // extern "C"
