// executor.cu -- the native ZeRO-1 bucket-flush executor.
//
// DeepSpeed issue #8700: DeepCompile's ZeRO-1 executor (Z1CustomOpExecutor)
// holds the owner map ("roots is therefore precomputed for the whole bucket
// before any collective is issued") and flushes each reduce bucket when it is
// full, with a probe line per flush.  This executor does the same on one GPU:
// at creation it validates everything and builds every bucket's launch plan
// (owners, delivered non-empty destinations, vector alignment, work units) and
// its probe counters; a flush is then one kernel launch with no per-call host
// work beyond copying the prebuilt plan into the launch.
//
// flush_all_from_host adds the host side of a step: the gradients arrive in
// pinned host memory and the reduced gradients go back to host memory.  The
// executor pipelines it over buckets on its own copy streams -- bucket b+1's
// host-to-device copy overlaps bucket b's flush, and each bucket's results
// start their device-to-host copy as soon as its flush ends -- and joins the
// caller's stream at the end.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"

struct dpred_executor {
    int world, in_dt, out_dt, pre_div;
    const char* grads;  // device [world, ld]
    int64_t ld;
    std::vector<int64_t> bucket_start;            // as given at creation
    std::vector<int64_t> start, size;             // per bucket: column range of the gradient rows
    std::vector<dpred::BuiltPlan> plans;          // per bucket
    std::vector<dpred_probe> probes;              // per bucket (flush_index filled per call)
    std::vector<std::vector<std::pair<char*, int64_t>>> written;  // per bucket: [device pointer, bytes] written
    std::vector<std::vector<dpred::Dest>> dests;  // per bucket: the delivered destinations the plan was built from
    // plans of the mapped host step, rebuilt when its host pointers change
    std::vector<dpred::BuiltPlan> mapped;
    std::vector<const void*> mapped_key;
    // launch overlap: bucket b+1's flush may start while bucket b's drains
    bool overlap_ok = false;         // the device buckets share no byte
    bool mapped_overlap_ok = false;  // the mapped plans share no byte
    bool overlap_on = true;          // dpred_executor_set_overlap
    bool in_place = false;           // results written back into the gradient rows
    void* workspace;
    size_t workspace_bytes;
    int64_t flushes = 0;
    // host pipeline resources, created on first use
    bool pipeline = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> ev_in, ev_out;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    std::mutex mu;
};

namespace {

int esz(int dt) { return dt == DPRED_BF16 ? 2 : 4; }

int setup_pipeline(dpred_executor* ex) {
    if (ex->pipeline) return DPRED_OK;
    cudaError_t e = cudaSuccess;
    e = cudaStreamCreateWithFlags(&ex->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ex->d2h, cudaStreamNonBlocking);
    const size_t nb = ex->plans.size();
    ex->ev_in.assign(nb, nullptr);
    ex->ev_out.assign(nb, nullptr);
    for (size_t b = 0; b < nb && e == cudaSuccess; ++b) {
        e = cudaEventCreateWithFlags(&ex->ev_in[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ex->ev_out[b], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ex->ev_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ex->ev_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return dpred::cuda_error(e, "executor stream/event creation");
    ex->pipeline = true;
    return DPRED_OK;
}

// True when no two flushes of the step can touch the same byte: the buckets'
// column ranges are disjoint, no two destination ranges overlap, and no
// destination lies inside the gradient array [grads, grads + grads_bytes).
// Only then may consecutive flushes overlap on the GPU.
bool buckets_independent(const std::vector<int64_t>& start, const std::vector<int64_t>& size,
                         const std::vector<std::vector<dpred::Dest>>& dests, int osz, const void* grads,
                         int64_t grads_bytes, int64_t row_bytes, int isz) {
    std::vector<std::pair<int64_t, int64_t>> cols;
    for (size_t b = 0; b < start.size(); ++b)
        if (size[b] > 0) cols.emplace_back(start[b], start[b] + size[b]);
    std::sort(cols.begin(), cols.end());
    for (size_t i = 1; i < cols.size(); ++i)
        if (cols[i].first < cols[i - 1].second) return false;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grads), g1 = g0 + (uintptr_t)grads_bytes;
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    for (size_t b = 0; b < dests.size(); ++b)
        for (const dpred::Dest& t : dests[b])
            if (t.numel > 0)
                for (void* p : t.ptrs) {
                    const uintptr_t a = reinterpret_cast<uintptr_t>(p), e = a + (uintptr_t)(t.numel * osz);
                    if (a < g1 && e > g0) {
                        // in place: the range must lie inside one row, within this
                        // bucket's own columns (which no other bucket reads or writes)
                        if (osz != isz || row_bytes <= 0 || a < g0 || e > g1) return false;
                        const uintptr_t off = a - g0;
                        if (off % (uintptr_t)isz) return false;
                        const int64_t col = (int64_t)((off % (uintptr_t)row_bytes) / (uintptr_t)isz);
                        if (col < start[b] || col + t.numel > start[b] + size[b]) return false;
                        continue;
                    }
                    r.emplace_back(a, e);
                }
    std::sort(r.begin(), r.end());
    uintptr_t end = 0;
    for (const auto& x : r) {
        if (x.first < end) return false;
        end = std::max(end, x.second);
    }
    return true;
}

int flush_one(dpred_executor* ex, int b, dpred_probe* probe, void* stream, bool pdl) {
    if (probe) {
        *probe = ex->probes[b];
        probe->flush_index = ex->flushes;
    }
    ex->flushes += 1;
    return dpred::launch_plan(ex->plans[b], ex->workspace, ex->workspace_bytes, static_cast<cudaStream_t>(stream), pdl);
}

// A new executor with its arguments checked; buckets are added by add_bucket.
int new_executor(int32_t world, int32_t in_dtype, int32_t out_dtype, int32_t pre_div, const void* grads, int64_t ld,
                 int32_t n_buckets, const int64_t* bucket_start, const int32_t* bucket_tasks, void* workspace,
                 size_t workspace_bytes, dpred_executor** out) {
    using namespace dpred;
    if (world < 1 || world > DPRED_MAX_WORLD) return set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n_buckets < 0 || (n_buckets > 0 && (!bucket_start || !bucket_tasks)))
        return set_error(DPRED_E_INVAL, "bad bucket list");
    if ((in_dtype != DPRED_BF16 && in_dtype != DPRED_F32) || (out_dtype != DPRED_BF16 && out_dtype != DPRED_F32))
        return set_error(DPRED_E_INVAL, "bad dtype");
    if (ld < 0) return set_error(DPRED_E_INVAL, "ld < 0");
    if (grads && reinterpret_cast<uintptr_t>(grads) % esz(in_dtype))
        return set_error(DPRED_E_ALIGN, "grads not aligned to its element size");
    for (int b = 0; b < n_buckets; ++b)
        if (bucket_tasks[b] < 0) return set_error(DPRED_E_INVAL, "bucket %d: negative task count", b);
    auto ex = new (std::nothrow) dpred_executor();
    if (!ex) return set_error(DPRED_E_INVAL, "out of host memory");
    ex->world = world;
    ex->in_dt = in_dtype;
    ex->out_dt = out_dtype;
    ex->pre_div = pre_div;
    ex->grads = static_cast<const char*>(grads);
    ex->ld = ld;
    ex->workspace = workspace;
    ex->workspace_bytes = workspace_bytes;
    ex->bucket_start.assign(bucket_start, bucket_start + n_buckets);
    *out = ex;
    return DPRED_OK;
}

// Bucket b: its tasks (for the column range) and its delivered destinations,
// already validated.  Builds the launch plan and records what the bucket writes.
int add_bucket(dpred_executor* ex, int b, const dpred_task* bt, int nt, std::vector<dpred::Dest>&& plan,
               const dpred_probe& pr) {
    using namespace dpred;
    const int64_t start = ex->bucket_start[b];
    int64_t width = 0;
    for (int t = 0; t < nt; ++t) width = std::max(width, bt[t].offset + bt[t].numel);
    if (start < 0 || start + width > ex->ld)
        return set_error(DPRED_E_SIZE, "bucket %d: columns [%lld, %lld) outside the row of %lld", b, (long long)start,
                         (long long)(start + width), (long long)ex->ld);
    if (width > 0 && ex->grads == nullptr) return set_error(DPRED_E_INVAL, "null grads");
    const int osz = esz(ex->out_dt);
    std::vector<std::pair<char*, int64_t>> wr;
    for (const Dest& d : plan)
        for (void* p : d.ptrs) {
            if (reinterpret_cast<uintptr_t>(p) % osz)
                return set_error(DPRED_E_ALIGN, "bucket %d: destination not aligned to its element size", b);
            if (d.numel > 0) wr.emplace_back(static_cast<char*>(p), d.numel * osz);
        }
    BuiltPlan bp;
    build_plan(ex->world, ex->in_dt, ex->grads + start * esz(ex->in_dt), ex->ld, ex->out_dt, ex->pre_div, plan, bp);
    if (bp.h.n_tasks > kInlineTasks || (int)bp.pool.size() > kInlineDst) {
        const size_t need = sizeof(TaskDesc) * bp.tasks.size() + ((bp.pool.size() * sizeof(void*) + 15) & ~(size_t)15);
        if (!ex->workspace || ex->workspace_bytes < need)
            return set_error(DPRED_E_SIZE, "bucket %d needs %zu bytes of workspace, got %zu", b, need,
                             ex->workspace_bytes);
    }
    ex->start.push_back(start);
    ex->size.push_back(width);
    ex->plans.push_back(std::move(bp));
    ex->probes.push_back(pr);
    ex->written.push_back(std::move(wr));
    ex->dests.push_back(std::move(plan));
    return DPRED_OK;
}

void finish_executor(dpred_executor* ex) {
    ex->overlap_ok = buckets_independent(ex->start, ex->size, ex->dests, esz(ex->out_dt), ex->grads,
                                         (int64_t)ex->world * ex->ld * esz(ex->in_dt), ex->ld * esz(ex->in_dt),
                                         esz(ex->in_dt));
}

void release(dpred_executor* ex) {
    if (ex->h2d) cudaStreamDestroy(ex->h2d);
    if (ex->d2h) cudaStreamDestroy(ex->d2h);
    for (auto e : ex->ev_in)
        if (e) cudaEventDestroy(e);
    for (auto e : ex->ev_out)
        if (e) cudaEventDestroy(e);
    if (ex->ev_start) cudaEventDestroy(ex->ev_start);
    if (ex->ev_done) cudaEventDestroy(ex->ev_done);
}

}  // namespace

extern "C" {

int dpred_host_mapped_pointer(const void* host, void** dev) {
    using namespace dpred;
    if (!host || !dev) return set_error(DPRED_E_INVAL, "null pointer");
    *dev = nullptr;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, host);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_error(e, "cudaPointerGetAttributes");
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr)
        return set_error(DPRED_E_INVAL, "%p is not page-locked host memory mapped into the device address space", host);
    *dev = a.devicePointer;
    return DPRED_OK;
}

int dpred_executor_create(int32_t world, int32_t in_dtype, int32_t out_dtype, int32_t pre_div, int32_t reduce_to_owner,
                          const int32_t* owner, int32_t n_params, const void* grads, int64_t ld, int32_t n_buckets,
                          const int64_t* bucket_start, const int32_t* bucket_tasks, const dpred_task* tasks,
                          void* const* dst, void* workspace, size_t workspace_bytes, dpred_executor** out) {
    using namespace dpred;
    if (!out) return set_error(DPRED_E_INVAL, "null executor output");
    *out = nullptr;
    dpred_executor* ex = nullptr;
    int rc = new_executor(world, in_dtype, out_dtype, pre_div, grads, ld, n_buckets, bucket_start, bucket_tasks,
                          workspace, workspace_bytes, &ex);
    if (rc) return rc;
    ex->in_place = dst == nullptr;
    if (ex->in_place && in_dtype != out_dtype) {
        delete ex;
        return set_error(DPRED_E_INVAL, "an in-place executor needs out_dtype == in_dtype");
    }
    const int isz = esz(in_dtype);
    int64_t t0 = 0, d0 = 0;
    for (int b = 0; b < n_buckets; ++b) {
        const int nt = bucket_tasks[b];
        const dpred_task* bt = tasks + t0;
        void* const* bd = ex->in_place ? nullptr : dst + d0;
        // Full validation through the public probe path (same rules as a flush).
        dpred_probe pr{};
        rc = dpred_flush_probe(world, bt, nt, owner, n_params, bd, reduce_to_owner, &pr);
        if (rc == DPRED_OK && ex->in_place) {
            std::vector<std::pair<int64_t, int64_t>> rg;
            for (int t = 0; t < nt; ++t)
                if (bt[t].numel > 0) rg.emplace_back(bt[t].offset, bt[t].offset + bt[t].numel);
            std::sort(rg.begin(), rg.end());
            for (size_t i = 1; i < rg.size() && rc == DPRED_OK; ++i)
                if (rg[i].first < rg[i - 1].second) rc = set_error(DPRED_E_SIZE, "bucket %d: in-place tasks overlap", b);
        }
        std::vector<Dest> plan(nt);
        for (int t = 0; t < nt && rc == DPRED_OK; ++t) {
            const int root = (reduce_to_owner && owner && owner[bt[t].param_id] >= 0) ? owner[bt[t].param_id] : -1;
            plan[t].src_off = bt[t].offset;
            plan[t].numel = bt[t].numel;
            for (int r = 0; r < world; ++r) {
                if (root >= 0 && r != root) continue;
                void* p = ex->in_place ? const_cast<char*>(static_cast<const char*>(grads)) +
                                             ((int64_t)r * ld + bucket_start[b] + bt[t].offset) * isz
                                       : bd[(int64_t)r * nt + t];
                if (p) plan[t].ptrs.push_back(p);
            }
        }
        if (rc == DPRED_OK) rc = add_bucket(ex, b, bt, nt, std::move(plan), pr);
        if (rc) {
            delete ex;
            return rc;
        }
        t0 += nt;
        d0 += (int64_t)world * nt;
    }
    finish_executor(ex);
    *out = ex;
    return DPRED_OK;
}

int dpred_executor_create_partitioned(int32_t world, int32_t in_dtype, int32_t out_dtype, int32_t pre_div,
                                      const void* grads, int64_t ld, int32_t n_buckets, const int64_t* bucket_start,
                                      const int32_t* bucket_tasks, const dpred_task* tasks,
                                      const int64_t* flat_offset, int32_t n_params, int64_t part_size,
                                      void* const* part_dst, void* workspace, size_t workspace_bytes,
                                      dpred_executor** out) {
    using namespace dpred;
    if (!out) return set_error(DPRED_E_INVAL, "null executor output");
    *out = nullptr;
    dpred_executor* ex = nullptr;
    int rc = new_executor(world, in_dtype, out_dtype, pre_div, grads, ld, n_buckets, bucket_start, bucket_tasks,
                          workspace, workspace_bytes, &ex);
    if (rc) return rc;
    int64_t t0 = 0;
    for (int b = 0; b < n_buckets; ++b) {
        const int nt = bucket_tasks[b];
        const dpred_task* bt = tasks + t0;
        dpred_probe pr{};
        std::vector<Dest> plan;
        rc = partitioned_plan(world, in_dtype, out_dtype, static_cast<const char*>(grads) + bucket_start[b] * esz(in_dtype),
                              ld, bt, nt, flat_offset, n_params, part_size, part_dst, plan, &pr);
        if (rc == DPRED_OK) rc = add_bucket(ex, b, bt, nt, std::move(plan), pr);
        if (rc) {
            delete ex;
            return rc;
        }
        t0 += nt;
    }
    finish_executor(ex);
    *out = ex;
    return DPRED_OK;
}

int dpred_executor_destroy(dpred_executor* ex) {
    if (!ex) return DPRED_OK;
    release(ex);
    delete ex;
    return DPRED_OK;
}

int dpred_executor_flush(dpred_executor* ex, int32_t bucket, dpred_probe* probe, void* stream) {
    using namespace dpred;
    if (!ex) return set_error(DPRED_E_INVAL, "null executor");
    if (bucket < 0 || bucket >= (int)ex->plans.size())
        return set_error(DPRED_E_INVAL, "bucket %d outside 0..%d", bucket, (int)ex->plans.size() - 1);
    return flush_one(ex, bucket, probe, stream, false);
}

int dpred_executor_flush_all(dpred_executor* ex, dpred_probe* probes, void* stream) {
    if (!ex) return dpred::set_error(DPRED_E_INVAL, "null executor");
    const bool pdl = ex->overlap_ok && ex->overlap_on;
    for (int b = 0; b < (int)ex->plans.size(); ++b) {
        // the first flush follows the caller's own work: never overlapped
        int rc = flush_one(ex, b, probes ? probes + b : nullptr, stream, pdl && b > 0);
        if (rc) return rc;
    }
    return DPRED_OK;
}

int dpred_executor_overlap_eligible(const dpred_executor* ex) {
    if (!ex) return dpred::set_error(DPRED_E_INVAL, "null executor");
    return ex->overlap_ok ? 1 : 0;
}

int dpred_executor_set_overlap(dpred_executor* ex, int32_t on) {
    if (!ex) return dpred::set_error(DPRED_E_INVAL, "null executor");
    const int prev = ex->overlap_on ? 1 : 0;
    ex->overlap_on = on != 0;
    return prev;
}

int dpred_executor_flush_all_from_host(dpred_executor* ex, const void* host_grads, int64_t host_ld, int32_t n_regions,
                                       void* const* region_dev, void* const* region_host, const int64_t* region_bytes,
                                       dpred_probe* probes, void* stream) {
    using namespace dpred;
    if (!ex) return set_error(DPRED_E_INVAL, "null executor");
    if (ex->in_place) return set_error(DPRED_E_INVAL, "host-buffer steps need destination buffers (in-place executor)");
    if (!host_grads || host_ld < 0) return set_error(DPRED_E_INVAL, "bad host gradients");
    if (n_regions < 0 || (n_regions > 0 && (!region_dev || !region_host || !region_bytes)))
        return set_error(DPRED_E_INVAL, "bad output regions");
    const int isz = esz(ex->in_dt);
    // every written destination range must lie inside one output region
    std::vector<std::vector<std::pair<int, std::pair<int64_t, int64_t>>>> copies(ex->plans.size());
    for (size_t b = 0; b < ex->plans.size(); ++b) {
        std::vector<std::pair<int64_t, int64_t>> span(n_regions, {INT64_MAX, -1});
        for (auto& w : ex->written[b]) {
            int hit = -1;
            for (int i = 0; i < n_regions && hit < 0; ++i) {
                const char* base = static_cast<const char*>(region_dev[i]);
                if (w.first >= base && w.first + w.second <= base + region_bytes[i]) hit = i;
            }
            if (hit < 0) return set_error(DPRED_E_INVAL, "bucket %zu writes outside every output region", b);
            const int64_t off = w.first - static_cast<const char*>(region_dev[hit]);
            span[hit].first = std::min(span[hit].first, off);
            span[hit].second = std::max(span[hit].second, off + w.second);
        }
        for (int i = 0; i < n_regions; ++i)
            if (span[i].second > span[i].first) copies[b].push_back({i, span[i]});
    }
    std::lock_guard<std::mutex> lock(ex->mu);
    int rc = setup_pipeline(ex);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(ex->ev_start, s);  // earlier work on the caller's stream comes first
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ex->h2d, ex->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ex->d2h, ex->ev_start, 0);
    for (size_t b = 0; b < ex->plans.size() && e == cudaSuccess; ++b) {
        // one contiguous copy per replica row: a pitched 2-D copy of a bucket
        // moves several times slower over the host link on this platform
        cudaStream_t cs = ex->h2d;
        const int64_t col = ex->start[b] * isz;
        for (int r = 0; r < ex->world && e == cudaSuccess; ++r)
            e = cudaMemcpyAsync(const_cast<char*>(ex->grads) + r * ex->ld * isz + col,
                                static_cast<const char*>(host_grads) + r * host_ld * isz + col,
                                (size_t)(ex->size[b] * isz), cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(ex->ev_in[b], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ex->ev_in[b], 0);
        if (e != cudaSuccess) break;
        rc = dpred_executor_flush(ex, (int)b, probes ? probes + b : nullptr, stream);
        if (rc) return rc;
        e = cudaEventRecord(ex->ev_out[b], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ex->d2h, ex->ev_out[b], 0);
        for (auto& c : copies[b]) {
            if (e != cudaSuccess) break;
            const int i = c.first;
            e = cudaMemcpyAsync(static_cast<char*>(region_host[i]) + c.second.first,
                                static_cast<const char*>(region_dev[i]) + c.second.first,
                                (size_t)(c.second.second - c.second.first), cudaMemcpyDeviceToHost, ex->d2h);
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(ex->ev_done, ex->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ex->ev_done, 0);  // the caller's stream completes last
    return e == cudaSuccess ? DPRED_OK : cuda_error(e, "executor host pipeline");
}

int dpred_executor_flush_all_mapped(dpred_executor* ex, const void* host_grads, int64_t host_ld, int32_t n_regions,
                                    void* const* region_dev, void* const* region_host, const int64_t* region_bytes,
                                    dpred_probe* probes, void* stream) {
    using namespace dpred;
    if (!ex) return set_error(DPRED_E_INVAL, "null executor");
    if (ex->in_place) return set_error(DPRED_E_INVAL, "host-buffer steps need destination buffers (in-place executor)");
    if (!host_grads || host_ld < 0) return set_error(DPRED_E_INVAL, "bad host gradients");
    if (reinterpret_cast<uintptr_t>(host_grads) % esz(ex->in_dt))
        return set_error(DPRED_E_ALIGN, "host gradients not aligned to their element size");
    if (n_regions < 0 || (n_regions > 0 && (!region_dev || !region_host || !region_bytes)))
        return set_error(DPRED_E_INVAL, "bad output regions");
    int64_t width = 0;
    for (size_t b = 0; b < ex->plans.size(); ++b) width = std::max(width, ex->start[b] + ex->size[b]);
    if (host_ld < width)
        return set_error(DPRED_E_SIZE, "host rows of %lld elements, the buckets span %lld", (long long)host_ld,
                         (long long)width);
    std::lock_guard<std::mutex> lock(ex->mu);
    std::vector<const void*> key{host_grads, reinterpret_cast<const void*>(host_ld)};
    for (int i = 0; i < n_regions; ++i) {
        key.push_back(region_dev[i]);
        key.push_back(region_host[i]);
        key.push_back(reinterpret_cast<const void*>(region_bytes[i]));
    }
    if (key != ex->mapped_key) {
        void* gdev = nullptr;
        int rc = dpred_host_mapped_pointer(host_grads, &gdev);
        if (rc) return rc;
        std::vector<char*> hdev(n_regions, nullptr);
        for (int i = 0; i < n_regions; ++i) {
            if (region_bytes[i] < 0) return set_error(DPRED_E_INVAL, "region %d: negative size", i);
            if (region_bytes[i] == 0) continue;
            void* d = nullptr;
            rc = dpred_host_mapped_pointer(region_host[i], &d);
            if (rc) return rc;
            hdev[i] = static_cast<char*>(d);
        }
        const int osz = esz(ex->out_dt);
        std::vector<BuiltPlan> plans(ex->plans.size());
        std::vector<std::vector<Dest>> mapped_dests;
        for (size_t b = 0; b < ex->plans.size(); ++b) {
            std::vector<Dest> d = ex->dests[b];
            for (Dest& t : d)
                for (void*& p : t.ptrs) {
                    const char* q = static_cast<const char*>(p);
                    int hit = -1;
                    for (int i = 0; i < n_regions && hit < 0; ++i) {
                        const char* base = static_cast<const char*>(region_dev[i]);
                        if (region_bytes[i] > 0 && q >= base && q + t.numel * osz <= base + region_bytes[i]) hit = i;
                    }
                    if (hit < 0) return set_error(DPRED_E_INVAL, "bucket %zu writes outside every output region", b);
                    p = hdev[hit] + (q - static_cast<const char*>(region_dev[hit]));
                }
            build_plan(ex->world, ex->in_dt, static_cast<const char*>(gdev) + ex->start[b] * esz(ex->in_dt), host_ld,
                       ex->out_dt, ex->pre_div, d, plans[b]);
            plans[b].ldg_only = true;
            mapped_dests.push_back(std::move(d));
        }
        // (host-step destinations never lie inside the host gradient rows: row_bytes 0)
        ex->mapped_overlap_ok = buckets_independent(ex->start, ex->size, mapped_dests, osz, gdev,
                                                    (int64_t)ex->world * host_ld * esz(ex->in_dt), 0,
                                                    esz(ex->in_dt));
        ex->mapped = std::move(plans);
        ex->mapped_key = std::move(key);
    }
    for (size_t b = 0; b < ex->mapped.size(); ++b) {
        if (probes) {
            probes[b] = ex->probes[b];
            probes[b].flush_index = ex->flushes;
        }
        ex->flushes += 1;
        const bool pdl = ex->mapped_overlap_ok && ex->overlap_on && b > 0;
        const int rc = launch_plan(ex->mapped[b], ex->workspace, ex->workspace_bytes, static_cast<cudaStream_t>(stream),
                                   pdl);
        if (rc) return rc;
    }
    return DPRED_OK;
}

}  // extern "C"
