/*
 * dpred.h -- C ABI of libdpred: data-parallel gradient reduction (ZeRO-1 bucket
 * flush, deferred accumulation, ReduceScatter / AllGather) on one GPU.
 *
 * The W data-parallel replicas are W rows of one array in device memory.  Each
 * "collective" of the pages becomes one streaming kernel over those rows:
 * Reduce -> written to one destination, AllReduce -> written to every
 * destination, ReduceScatter / AllGather -> reduce-and-shard / copy layouts.
 *
 * Pages this interface follows (cited by title and section):
 *  [DS] DeepSpeed issue #8700 "[REQUEST] DeepCompile ZeRO-1: reduce-to-owner
 *       instead of AllReduce".
 *  [MT] MaxText PR #5099 "Defer the data-parallel gradient all-reduce to
 *       update() under gradient accumulation".
 *  [AG] "AllGather" (tier6-model interconnect notes, 集合通信 / all-gather).
 *
 * Conventions shared by every call:
 *  - Return value: DPRED_OK (0) or a negative DPRED_E_* code.  Nothing aborts
 *    or traps.  dpred_last_error() gives this thread's message for the last
 *    failure.  Arguments are validated before any device work is enqueued; a
 *    call that fails validation enqueues nothing.
 *  - Memory: the caller owns all memory; the library allocates no device
 *    memory.  "device" pointers are CUDA device (or managed) addresses,
 *    "host" pointers are ordinary process memory read during the call only.
 *  - Element types: DPRED_BF16 (bfloat16, 2 bytes) and DPRED_F32 (4 bytes).
 *    Every data pointer must be aligned to its element size (DPRED_E_ALIGN);
 *    16-byte alignment is not required but enables the vectorised path.
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *    Device work is enqueued on it and the call returns without waiting.
 *  - Stream capture: a call whose plan goes to a caller workspace (the
 *    flush, the partitioned flush and the relayout when their
 *    *_workspace_bytes() is nonzero) uploads that plan from host memory, and
 *    refuses a stream that is being captured into a CUDA graph with
 *    DPRED_E_INVAL before enqueuing anything: the captured copy would read
 *    the host plan again at every replay.
 *  - Arithmetic of every reduction: each term is widened to fp32, optionally
 *    pre-divided by the number of ranks (IEEE division), and the terms are
 *    summed in fp32 in rank order 0, 1, ..., W-1 starting from the rank-0
 *    term; the sum is rounded once to the output type (bf16: round to
 *    nearest, ties to even).  The order never depends on the launch shape, so
 *    results are bitwise reproducible.
 */
#ifndef DPRED_H
#define DPRED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DPRED_OK 0
#define DPRED_E_INVAL (-1)    /* bad argument (null pointer, bad dtype, negative size, ...) */
#define DPRED_E_ALIGN (-2)    /* a pointer is not aligned to its element size */
#define DPRED_E_SIZE (-3)     /* sizes inconsistent (range outside a row, M % N != 0, workspace too small) */
#define DPRED_E_MISMATCH (-4) /* checked mode: destinations disagree with the owner map */
#define DPRED_E_CUDA (-5)     /* a CUDA runtime call failed */
#define DPRED_E_TIMEOUT (-6)  /* a device-side bounded wait gave up (reported by dpred_device_status) */
#define DPRED_E_BOUNDS (-7)   /* checked build: a kernel access failed its bounds test and was skipped
                                 (reported by dpred_device_status) */

/* element types */
#define DPRED_BF16 0
#define DPRED_F32 1

#define DPRED_MAX_WORLD 64

/* One parameter group ([DS] "Design points": param groups; groups reduced
 * over another communicator are excluded from the owner map). */
typedef struct {
    int32_t comm_size;          /* ranks of the group's communicator */
    int32_t n_params;           /* parameters in the group */
    const int32_t* comm_ranks;  /* host [comm_size]: group rank -> data-parallel rank; NULL = identity */
    const int64_t* numel;       /* host [n_params]: sizes in the group's flat (model) order */
} dpred_group;

/* One task of a reduce bucket: one whole parameter gradient ([DS] "Describe
 * alternatives you've considered": buckets are assembled in gradient-arrival
 * order, one full-parameter task each).  24 bytes. */
typedef struct {
    int32_t param_id;  /* index into the owner map */
    int32_t reserved;  /* must be 0 */
    int64_t offset;    /* element offset of the task inside every bucket row */
    int64_t numel;     /* elements */
} dpred_task;

/* Probe counters of one flush ([DS] "reduce_probe" and the printed probe
 * line).  discarded% of rank r = 100 * (reduced_elems - kept_elems[r]) /
 * reduced_elems; owner% = 100 * owner_elems / reduced_elems. */
typedef struct {
    int64_t flush_index;    /* in: caller's flush counter, copied through unchanged */
    int64_t tasks;          /* tasks in the bucket */
    int64_t reduced_elems;  /* sum of task sizes */
    int64_t owner_tasks;    /* tasks that took the reduce-to-owner path */
    int64_t owner_elems;    /* their elements */
    int64_t kept_elems[DPRED_MAX_WORLD]; /* per rank: elements of tasks whose destination is non-empty */
} dpred_probe;

const char* dpred_last_error(void);
const char* dpred_version(void);
/* 1 in the checked build (compiled with -DDPRED_CHECKED=1, loaded when the
 * environment sets DPRED_CHECKED=1): every global load and store of the flush
 * kernels (flush, ReduceScatter, the executor's steps; both kernel families)
 * is first tested against the task it belongs to -- source vector inside the
 * task's aligned body and inside the row, destination element range inside
 * the task -- and a failed test records DPRED_E_BOUNDS in the device error
 * word and skips the access.  0 in the default build, where the tests compile
 * away.  No counterpart in the pages. */
int dpred_checked_build(void);

/*
 * Owner map.  [DS] "Design points" ("Owner map costs nothing to build",
 * "Partial parameters keep AllReduce", "No native flag", "Parameter groups
 * reduced over a different communicator are skipped").
 *
 * Each group's flat space of T elements is cut into comm_size contiguous
 * partitions of ceil(T / comm_size) elements (the last one shorter).  A
 * parameter covering [s, e) is held by partitions lo = s / P .. hi = (e-1) / P.
 * owner[p] = lo when lo == hi, the group is eligible and reduce_to_owner != 0;
 * otherwise -1 (AllReduce).  Eligible: comm_size == world and comm_ranks[i] == i.
 * For an ineligible group owner = -1 and every data-parallel rank is treated
 * as a holder (holder_lo = 0, holder_hi = world - 1); a zero-size parameter
 * has owner = holder_lo = holder_hi = -1.  The result does not depend on
 * `rank` (the map is identical on every rank).
 *
 * Host only, synchronous.  Outputs (host, caller-allocated) are indexed by
 * parameter in group order then flat order: owner, holder_lo, holder_hi
 * [sum n_params]; *n_owned = parameters with an owner, *n_total = all
 * parameters (the "k/total gradients reduce to one rank" report).
 * Errors: DPRED_E_INVAL for world outside 1..DPRED_MAX_WORLD, rank outside
 * 0..world-1, negative sizes or null pointers.
 */
int dpred_build_owner_map(int32_t world, int32_t rank, const dpred_group* groups, int32_t n_groups,
                          int32_t reduce_to_owner, int32_t* owner, int32_t* holder_lo, int32_t* holder_hi,
                          int32_t* n_owned, int32_t* n_total);

/*
 * Digest of an owner map (64-bit FNV-1a over n_params and the owner,
 * holder_lo and holder_hi arrays, host).  [DS] "Design points": the map must
 * be identical on every rank, because it decides which collective each bucket
 * entry uses and every rank has to issue the same sequence.  Ranks exchange
 * this digest to detect one built from inconsistent metadata before any flush.
 */
uint64_t dpred_owner_map_digest(int32_t n_params, const int32_t* owner, const int32_t* holder_lo,
                                const int32_t* holder_hi);

/*
 * The owner map of one parameter group, computed on the device (for an
 * executor whose parameter table lives in device memory).  Same rule and
 * results as dpred_build_owner_map for a single group: numel (device, int64
 * [n_params]) in flat order; comm_ranks (device, int32 [comm_size]) or NULL
 * for the identity; outputs owner / holder_lo / holder_hi (device, int32
 * [n_params]) and counts (device, int32 [2]: n_owned, n_total).  One CTA:
 * warp-shuffle reduction of the sizes for the partition size, warp-shuffle
 * exclusive scan for the flat starts, warp ballots for the owned count.
 * Errors: DPRED_E_INVAL, DPRED_E_ALIGN, DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_build_owner_map_device(int32_t world, int32_t n_params, const int64_t* numel, int32_t comm_size,
                                 const int32_t* comm_ranks, int32_t reduce_to_owner, int32_t* owner,
                                 int32_t* holder_lo, int32_t* holder_hi, int32_t* counts, void* stream);

/*
 * Probe counters of a flush from its metadata alone, without launching
 * anything ([DS] "reduce_probe": size the win before turning the path on).
 * Arguments as for dpred_flush_bucket.  kept_elems[r] sums the tasks whose
 * rank-r destination dst[r * n_tasks + t] is non-NULL; with dst == NULL (in
 * place) it sums the tasks delivered to row r.  probe->flush_index is left as
 * the caller set it.  Host only.
 */
int dpred_flush_probe(int32_t world, const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                      int32_t n_params, void* const* dst, int32_t reduce_to_owner, dpred_probe* probe);

/*
 * The probe line of one flush for one rank ([DS] "Is your feature request
 * related to a problem? Please describe.": the reduce_probe log line, e.g.
 * "[dc-probe][r0] flushReduceBucket #3 dtype=BFloat16 tasks=118
 * reduced_elems=52428800 kept_elems=6553600 discarded=87.5% pre_div=1
 * owner_tasks=0 owner_elems=0 (0.0%)").  discarded% = 100 * (reduced_elems -
 * kept_elems[rank]) / reduced_elems and owner% = 100 * owner_elems /
 * reduced_elems, both with one decimal (0.0 for an empty flush); dtype names
 * the gradient type ("BFloat16" or "Float").  probe (host) holds the counters
 * of dpred_flush_probe or dpred_flush_bucket; the NUL-terminated line is
 * written to buf (host, buf_bytes bytes; 256 always suffice).  Synchronous,
 * no device work.  Errors: DPRED_E_INVAL (null pointer, world outside
 * 1..DPRED_MAX_WORLD, rank outside 0..world-1, bad dtype), DPRED_E_SIZE
 * (buffer too small; buf then holds a truncated line).
 */
int dpred_probe_format(const dpred_probe* probe, int32_t world, int32_t rank, int32_t dtype, int32_t pre_div,
                       char* buf, size_t buf_bytes);

/*
 * Device workspace (bytes) that dpred_flush_bucket may need for a bucket of
 * n_tasks tasks at this world size.  Buckets of up to 128 tasks with up to
 * 512 written destinations travel inside the kernel launch and need none; for
 * larger ones the task table is copied (host -> device, from pageable memory,
 * so such a call waits for the copy to be staged) into the workspace.
 */
size_t dpred_flush_workspace_bytes(int32_t world, int32_t n_tasks);

/*
 * ZeRO-1 bucket flush.  [DS] "Describe the solution you'd like" (for a
 * parameter inside one partition, reduce to the single rank that keeps it:
 * same reduction, same operand order, one destination instead of ws), design
 * points "Partial parameters keep AllReduce", "Copy-out is unchanged and
 * still correct" and "Summation semantics untouched" (pre-division by the
 * world size before the sum), and the copy-out loop that skips empty buffers.
 *
 * grads (device) is the bucket: `world` rows of in_dtype elements, row r
 * starting at element r * ld.  Task t reduces elements
 * [offset, offset + numel) of every row.  root(t) = owner[param_id] when
 * reduce_to_owner != 0 and owner != NULL and it is >= 0, else -1.  The
 * reduced values go to rank root(t) only (root >= 0) or to every rank
 * (root == -1, the AllReduce fallback), and to a delivered rank r only if
 * its destination is non-empty:
 *  - dst != NULL: host array [world * n_tasks] of device pointers;
 *    dst[r * n_tasks + t] is rank r's buffer for task t (numel out_dtype
 *    elements) or NULL for an empty buffer.  Buffers of ranks that are not
 *    delivered are never touched.
 *  - dst == NULL: in place; the result overwrites the task's range in the
 *    delivered rows of grads.  out_dtype must equal in_dtype and tasks must
 *    not overlap.
 * owner: host [n_params] or NULL (no owners: AllReduce everything, the
 * flag-off path).  pre_div != 0 divides every term by world.  flags (an OR
 * of the DPRED_FLUSH_* bits below, 0 for none):
 *  - DPRED_FLUSH_CHECKED additionally verifies that an owner task has no
 *    non-NULL destination on a rank other than its owner (DPRED_E_MISMATCH);
 *  - DPRED_FLUSH_OVERLAP is the caller's promise that this flush shares no
 *    byte with the work enqueued on `stream` just before it (normally the
 *    previous bucket's flush): neither reads what that work writes nor
 *    writes what it reads or writes.  The flush may then start on the SMs
 *    that the previous flush's last wave leaves idle (programmatic dependent
 *    launch); it still completes after that flush, so the stream's order of
 *    completion is unchanged.  Plans that do not fit inside the launch
 *    (dpred_flush_workspace_bytes() > 0) ignore the bit.  A promise that
 *    does not hold makes the results undefined.
 * probe (host, may be NULL) receives the counters of dpred_flush_probe.
 * workspace (device, may be NULL when dpred_flush_workspace_bytes() is 0) of
 * workspace_bytes bytes.
 * Repeated calls: each thread keeps the validated plans and counters of its
 * 16 most recent distinct calls, keyed on every input byte (scalars, the task
 * table, owner[param_id] of each task and the destination table); a call
 * whose inputs equal one of them skips validation and planning.  Pointer
 * values are compared, never the memory behind them.
 * Asynchronous on `stream`; grads, dst buffers and workspace must stay valid
 * until the work completes.  Errors: DPRED_E_INVAL (including unknown flag
 * bits), DPRED_E_ALIGN, DPRED_E_SIZE (a task outside [0, ld), overlapping
 * in-place tasks, workspace too small), DPRED_E_MISMATCH, DPRED_E_CUDA.
 */
#define DPRED_FLUSH_CHECKED 1
#define DPRED_FLUSH_OVERLAP 2
int dpred_flush_bucket(int32_t world, int32_t in_dtype, void* grads, int64_t ld, const dpred_task* tasks,
                       int32_t n_tasks, const int32_t* owner, int32_t n_params, int32_t out_dtype, void* const* dst,
                       int32_t pre_div, int32_t reduce_to_owner, int32_t flags, dpred_probe* probe,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free bucket flush.  The pages have no counterpart to this entry
 * point; it serves callers that cannot allocate device memory: runtimes that
 * carve all device memory out of a fixed budget up front and have none left
 * to lend, and plug-ins that live inside another framework's allocator and
 * may not allocate device memory of their own.
 *
 * Same arguments and results as dpred_flush_bucket, minus the workspace.  A
 * bucket whose task table does not fit inside the launch uses a scratch
 * array of DPRED_NOALLOC_SCRATCH_BYTES (1 MiB) compiled into the library;
 * every GPU that loads the library holds that array until the process exits.
 * Buckets with dpred_flush_workspace_bytes(world, n_tasks) above
 * DPRED_NOALLOC_SCRATCH_BYTES are rejected with DPRED_E_SIZE before anything
 * is enqueued.  The call allocates no device memory.
 * Set-up: the first call made on a device looks up the scratch array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.
 * Sharing: all calls use the same scratch array, and each call overwrites the
 * part it uses (nothing in it has to start at zero).  Calls whose work can
 * overlap on the GPU -- on different streams without ordering between them --
 * race on the array; issue them on one stream or order them with events.
 */
#define DPRED_NOALLOC_SCRATCH_BYTES (1u << 20)
int dpred_flush_bucket_noalloc(int32_t world, int32_t in_dtype, void* grads, int64_t ld, const dpred_task* tasks,
                               int32_t n_tasks, const int32_t* owner, int32_t n_params, int32_t out_dtype,
                               void* const* dst, int32_t pre_div, int32_t reduce_to_owner, int32_t flags,
                               dpred_probe* probe, void* stream);

/*
 * The ZeRO-1 bucket-flush executor.  [DS] names Z1CustomOpExecutor::
 * flushReduceBucket, which precomputes the roots of a whole bucket before
 * issuing it and flushes each bucket when it is full.  An executor is bound
 * to one gradient array (grads, device, [world, ld] of in_dtype) and to its
 * buckets: bucket b covers columns [bucket_start[b], ...) with bucket_tasks[b]
 * tasks, taken in order from the concatenated `tasks`, and its destination
 * table of world * bucket_tasks[b] pointers, taken in order from the
 * concatenated `dst` (same meaning as in dpred_flush_bucket; NULL = empty
 * buffer).  dpred_executor_create validates every bucket with the flush's
 * rules and prebuilds every launch plan and probe, so a flush is one kernel
 * launch.  workspace (device) must hold the largest plan beyond the inline
 * limit (dpred_flush_workspace_bytes) for as long as the executor is used.
 * The executor keeps the flush counter of the probe lines.  Host memory only;
 * no device memory is allocated.
 *   dpred_executor_flush:     flush one bucket on `stream` (probe may be NULL).
 *   dpred_executor_flush_all: flush every bucket in order (probes: NULL or
 *                             one per bucket).
 *   dpred_executor_flush_all_from_host: one step with host buffers.  The
 *     bucket columns of host_grads ([world, host_ld], pinned host memory)
 *     are copied into grads, each bucket is flushed, and everything each
 *     bucket wrote is copied back into host memory: the destinations must lie
 *     in the n_regions device regions region_dev[i] (region_bytes[i] bytes),
 *     mirrored by pinned host regions region_host[i] at the same offsets.
 *     The copies run on the executor's own streams, pipelined over buckets
 *     (bucket b+1 arrives while bucket b is reduced; bucket b's results
 *     leave as soon as it is done); `stream` waits for its earlier work first
 *     and finishes after the last copy.  The first call creates the streams
 *     and events.  Not re-entrant for one executor.
 *   dpred_executor_flush_all_mapped: the same step with the same arguments:
 *     every destination byte a flush writes lands at the same place in the
 *     host regions (host bytes no destination covers stay untouched).  But
 *     nothing is staged in device memory: the flush kernels read the bucket
 *     columns of host_grads and
 *     write the reduced gradients into the host regions directly, over the
 *     host link (the memory must be pinned and mapped, see
 *     dpred_host_mapped_pointer).  grads and the device regions are neither
 *     read nor written; the device regions only say where in the host
 *     regions each result goes.  One launch per bucket on `stream`, in order;
 *     no extra streams.  The plans for a set of host pointers are built on
 *     the first call that uses them and reused while they stay the same.
 *     host_ld must cover every bucket's columns (DPRED_E_SIZE).
 *   dpred_executor_destroy:   release the executor (after its work is done).
 * In place: dst == NULL makes every flush write its delivered results back
 * into the gradient rows themselves, as dpred_flush_bucket does without a
 * destination table (row owner(t) for an owned parameter, every row for an
 * AllReduce one).  It needs out_dtype == in_dtype (else DPRED_E_INVAL) and
 * no two tasks of a bucket overlapping (else DPRED_E_SIZE).  Its probes
 * count what each row received.  The host-buffer steps need destination
 * buffers and return DPRED_E_INVAL on an in-place executor.
 */
typedef struct dpred_executor dpred_executor;
int dpred_executor_create(int32_t world, int32_t in_dtype, int32_t out_dtype, int32_t pre_div, int32_t reduce_to_owner,
                          const int32_t* owner, int32_t n_params, const void* grads, int64_t ld, int32_t n_buckets,
                          const int64_t* bucket_start, const int32_t* bucket_tasks, const dpred_task* tasks,
                          void* const* dst, void* workspace, size_t workspace_bytes, dpred_executor** out);
/*
 * The same executor over partitioned flushes (the ZeRO-2 form of rows f1/f3,
 * see dpred_flush_bucket_partitioned): bucket b's tasks are cut at the
 * partition boundaries of the flat space (flat_offset[param_id], partitions of
 * part_size elements) and every piece is written into its rank's partition
 * buffer part_dst[rank] (device, part_size elements of out_dtype; NULL =
 * that rank's partition is not kept).  Every other call above works on it
 * unchanged: flush, flush_all (with launch overlap), the two host-buffer
 * steps (the regions are then the partition buffers), destroy.  The probes
 * count as the partitioned flush's do.  Errors as in
 * dpred_flush_bucket_partitioned and dpred_executor_create.
 */
int dpred_executor_create_partitioned(int32_t world, int32_t in_dtype, int32_t out_dtype, int32_t pre_div,
                                      const void* grads, int64_t ld, int32_t n_buckets, const int64_t* bucket_start,
                                      const int32_t* bucket_tasks, const dpred_task* tasks,
                                      const int64_t* flat_offset, int32_t n_params, int64_t part_size,
                                      void* const* part_dst, void* workspace, size_t workspace_bytes,
                                      dpred_executor** out);
int dpred_executor_flush(dpred_executor* ex, int32_t bucket, dpred_probe* probe, void* stream);
int dpred_executor_flush_all(dpred_executor* ex, dpred_probe* probes, void* stream);
/*
 * Launch overlap (no counterpart in the pages).  When no two buckets of the
 * executor can touch the same byte (disjoint column ranges, no two
 * destination ranges overlapping, no destination inside the gradient array
 * except in place, inside its own bucket's columns of one row;
 * checked once at creation, and for the mapped step whenever its host
 * pointers change), dpred_executor_flush_all and _flush_all_mapped launch
 * every flush after the first with programmatic stream serialisation: it
 * starts on the SMs that the previous flush's last wave leaves idle, and it
 * still completes after the previous flush, so work queued later on the
 * stream sees every bucket done.  The first flush of a call never overlaps
 * the caller's earlier work.  on = 0 turns it off; on by default.  Returns
 * the previous setting (0/1), or DPRED_E_INVAL for a null executor.
 */
int dpred_executor_set_overlap(dpred_executor* ex, int32_t on);
/* 1 when the executor's device buckets passed that check, 0 when not,
 * DPRED_E_INVAL for a null executor.  Host only. */
int dpred_executor_overlap_eligible(const dpred_executor* ex);
int dpred_executor_flush_all_from_host(dpred_executor* ex, const void* host_grads, int64_t host_ld, int32_t n_regions,
                                       void* const* region_dev, void* const* region_host, const int64_t* region_bytes,
                                       dpred_probe* probes, void* stream);
int dpred_executor_flush_all_mapped(dpred_executor* ex, const void* host_grads, int64_t host_ld, int32_t n_regions,
                                    void* const* region_dev, void* const* region_host, const int64_t* region_bytes,
                                    dpred_probe* probes, void* stream);
int dpred_executor_destroy(dpred_executor* ex);

/*
 * Partitioned flush: every rank receives exactly its optimizer partition's
 * slice of the reduced bucket.  [DS] "Describe alternatives you've considered"
 * (ncclReduceScatter over the bucket, "the better end state", same traffic
 * class as reduce-to-owner) and "Follow-up" (ZeRO-2 registers real buffers
 * with offsets, so the destination is a slice of the rank's partition, not a
 * full-parameter buffer).  Here it is one fused pass over the arrival-order
 * bucket; no relayout is needed.
 *
 * grads, ld, tasks, pre_div: as for dpred_flush_bucket.  flat_offset (host,
 * [n_params]) is each parameter's start in its group's flat space;
 * part_size = ceil(T / world) elements per partition.  Element k of task t
 * (flat position f = flat_offset[param_id] + k) is reduced and written to
 * part_dst[r][f - r * part_size] with r = f / part_size; part_dst (host,
 * [world]) holds device pointers to the ranks' partition buffers (part_size
 * elements of out_dtype; NULL = that rank receives nothing).  A parameter
 * straddling a boundary is split there: each holder receives only its own
 * slice.  probe (may be NULL): tasks, reduced_elems, owner_tasks/owner_elems
 * = tasks lying inside one partition, kept_elems[r] = elements delivered to
 * rank r.  Workspace: dpred_flush_workspace_bytes(world, n_tasks + world - 1)
 * bytes suffice.  Errors: DPRED_E_INVAL, DPRED_E_ALIGN, DPRED_E_SIZE (a task
 * outside the row or the world's partitions, overlapping tasks, workspace too
 * small), DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_flush_bucket_partitioned(int32_t world, int32_t in_dtype, const void* grads, int64_t ld,
                                   const dpred_task* tasks, int32_t n_tasks, const int64_t* flat_offset,
                                   int32_t n_params, int64_t part_size, int32_t out_dtype, void* const* part_dst,
                                   int32_t pre_div, dpred_probe* probe, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * Bucket relayout pass: the copy that ncclReduceScatter over an arrival-order
 * bucket needs first ([DS] "Describe alternatives you've considered").  Every
 * replica row q of grads is rewritten rank-major into out (device,
 * [world, out_ld], out_ld >= world * seg): out[q][r * seg + j] = the j-th
 * element, in flat order, of the bucket's elements that lie in partition r.
 * seg_used (host, [world]) receives each run's length; out elements past a
 * run are not written.  dpred_reduce_scatter(world, world * seg, ...) of out
 * then gives rank r its reduced run, identical to what
 * dpred_flush_bucket_partitioned writes.  Arguments as for the partitioned
 * flush; the bucket's elements within one partition must form one contiguous
 * flat run (true for whole-parameter buckets of consecutive parameters).  A
 * pure byte copy.  Workspace: dpred_bucket_relayout_workspace_bytes(world,
 * n_tasks).  Asynchronous on `stream`.
 */
size_t dpred_bucket_relayout_workspace_bytes(int32_t world, int32_t n_tasks);
int dpred_bucket_relayout(int32_t world, int32_t dtype, const void* grads, int64_t ld, const dpred_task* tasks,
                          int32_t n_tasks, const int64_t* flat_offset, int32_t n_params, int64_t part_size, int64_t seg,
                          void* out, int64_t out_ld, int64_t* seg_used, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * Replica-local gradient accumulation with one cross-replica reduction per
 * optimizer step.  [MT] "What" (cotangents come out unreduced, a per-replica
 * partial sum that accumulates replica-locally across micro-batches; update()
 * emits the single cross-replica all-reduce).
 *
 * acc (device, fp32) and g (device, g_dtype) are [world, n], row-contiguous.
 * For every replica r and element k:  a = first ? g[r][k] : acc[r][k] + g[r][k].
 *  - finalize == 0: acc[r][k] = a.
 *  - finalize != 0: total[k] = (a[0] + a[1] + ... + a[world-1]) * scale (rank
 *    order, fp32), total (device, fp32, [n]); acc is not written (the
 *    accumulator is consumed by the reduction), so the last micro-batch's add
 *    and the cross-replica reduction are one pass.
 * scale multiplies the finished sum (e.g. 1 / denominator; 1.0 leaves it
 * unchanged).  Asynchronous on `stream`.  Errors: DPRED_E_INVAL (null
 * pointer, bad dtype, n < 0, world outside 1..DPRED_MAX_WORLD),
 * DPRED_E_ALIGN, DPRED_E_CUDA.
 */
int dpred_accumulate_microbatch(int32_t world, int64_t n, float* acc, int32_t g_dtype, const void* g,
                                int32_t first, int32_t finalize, float scale, float* total, void* stream);

/*
 * Accumulator checkpoints.  [MT] "What else had to change", "Accumulator
 * lifetime": a checkpoint holds the reduced total, so saving runs the pending
 * cross-replica all-reduce; restoring moves a total back onto the unreduced
 * form by leaving it on one replica and zeros on the rest, so that the next
 * deferred reduction reproduces it.
 *   dpred_accumulator_save:    total[k] = acc[0][k] + ... + acc[W-1][k]
 *                              (rank order, fp32, no scale); acc is not changed.
 *   dpred_accumulator_restore: acc[0][k] = total[k]; acc[r][k] = +0 for r > 0.
 * acc (device) is [world, n] fp32 row-contiguous, total (device) is [n] fp32.
 * Restore followed by save returns the total bit for bit (a -0 becomes +0).
 * Errors: DPRED_E_INVAL, DPRED_E_ALIGN, DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_accumulator_save(int32_t world, int64_t n, const float* acc, float* total, void* stream);
int dpred_accumulator_restore(int32_t world, int64_t n, float* acc, const float* total, void* stream);

/*
 * ReduceScatter.  [AG] "与 ReduceScatter 的对偶关系" (duality table: M
 * elements in per node, M/N out per node, reduce then shard).
 * in (device) is [n_nodes, m_elems] of in_dtype; out (device) is
 * [n_nodes, m_elems / n_nodes] of out_dtype; out[i][k] is the reduction of
 * in[0..N-1][i * S + k], S = m_elems / n_nodes (pre_div divides every term by
 * n_nodes).  Errors: DPRED_E_SIZE when m_elems % n_nodes != 0, DPRED_E_INVAL,
 * DPRED_E_ALIGN, DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_reduce_scatter(int32_t n_nodes, int64_t m_elems, int32_t in_dtype, const void* in, int32_t out_dtype,
                         void* out, int32_t pre_div, void* stream);

/*
 * AllGather.  [AG] "语义定义" (eq. ag-semantic-output: every node ends with
 * B_i = [A_0, A_1, ..., A_{N-1}]) and "Ring AllGather" (the N=4 table: after
 * the ring schedule node i holds [A_i, A_{i-1}, ..., A_{i-N+1}], indices mod N).
 * in (device) is [n_nodes, shard_elems] (row j = A_j); out (device) is
 * [n_nodes, n_nodes * shard_elems]:
 *   order 0 (canonical): out[i][c * S + k] = in[c][k]
 *   order 1 (ring):      out[i][c * S + k] = in[(i - c) mod N][k]
 * A bit copy: the element type only sets the element size.  Errors:
 * DPRED_E_INVAL (order not 0/1, ...), DPRED_E_ALIGN, DPRED_E_CUDA.
 * Asynchronous on `stream`.
 */
int dpred_allgather(int32_t n_nodes, int64_t shard_elems, int32_t dtype, const void* in, void* out, int32_t order,
                    void* stream);

/*
 * Kernel family used by later dpred_flush_bucket, dpred_reduce_scatter and
 * dpred_allgather calls in this process (a tuning knob; results are
 * bit-identical either way):
 *   0 auto (the default: the family measured fastest on GB300 for each call:
 *     register streaming for the flush and ReduceScatter, TMA for AllGather),
 *   1 register streaming: every thread keeps one 16-byte load per replica row
 *     (two at world 2, 3 and 4) for the flush, or per shard for AllGather, in
 *     flight and stores from registers,
 *   2 TMA staging: the flush has one thread per SM stream 4 KB row tiles into a
 *     ring of shared-memory stages with cp.async.bulk (mbarrier-counted) while
 *     eight warps reduce from shared memory (world in {2, 4, 8, 16} only;
 *     other world sizes use family 1); AllGather bulk-loads 16 KB shard tiles
 *     into shared memory once and bulk-stores each to its N destinations
 *     (16-byte aligned shards only).
 * Returns the previous setting, or DPRED_E_INVAL.  Not thread-safe against
 * concurrent flush calls.
 */
int dpred_set_flush_path(int32_t path);

/*
 * Kernel form of later dpred_allgather calls in this process (a tuning knob;
 * every form writes the same bytes):
 *   0 auto: form 1 when dpred_set_flush_path selected register streaming,
 *     else form 5,
 *   1 register streaming (16-byte loads and streaming stores, shard by shard),
 *   2 bulk copies, one issuing thread per SM: 16 KB shard tiles bulk-loaded
 *     into an 8-stage shared-memory ring and bulk-stored to the N rows,
 *   3 bulk copies, four issuing warps per SM, each with its own 6-stage ring
 *     of 8 KB tiles and its own bulk group,
 *   4 staged warp stores: one thread bulk-loads 16 KB tiles into an 8-stage
 *     ring, eight warps store each tile to the N rows with 16-byte streaming
 *     stores,
 *   5 bulk copies with rows skewed in time: one issuing thread per SM keeps
 *     the last min(N, 8) tiles staged (16 KB tiles, 12 stages) and in each
 *     step stores tile q - (i mod 8) to row i, so that concurrent stores to
 *     neighbouring rows are not a whole row apart,
 *   6 form 5 with 8 KB tiles and 20 stages.
 * Forms 2-6 need 16-byte aligned rows (else form 1 runs).  Returns the
 * previous form, or DPRED_E_INVAL.  Not thread-safe against concurrent calls.
 */
int dpred_set_allgather_form(int32_t form);

/*
 * AllGather schedules, executed step by step.  [AG] "Ring AllGather" (N-1
 * steps; in step s every node forwards to its right neighbour the chunk it
 * received in step s-1), the bidirectional ring (eq. ag-bidir-ring:
 * ceil((N-1)/2) steps; in step s node i receives chunk i-s from its left and
 * chunk i+s from its right neighbour) and "Recursive Doubling AllGather"
 * (N = 2^k; log2 N steps; in step j node i receives everything node
 * i xor 2^(j-1) holds).  The N node buffers are the rows of bufs (device,
 * [N, N * shard_elems]); slot c of row i holds one shard.  Layouts: ring
 * lists in ring order (slot c of node i = A_{(i-c) mod N}, as the page's N=4
 * table and dpred_allgather order 1); bidirectional ring and recursive
 * doubling keep every chunk at its own index (order 0).
 *   dpred_allgather_schedule_steps: the number of steps, or DPRED_E_INVAL.
 *   dpred_allgather_schedule_init:  copies shard i of in ([N, shard_elems])
 *                                   into node i's first slot (ring) or slot i.
 *   dpred_allgather_schedule_step:  one step (1 <= step <= steps): one kernel
 *                                   launch moving exactly the chunks that the
 *                                   schedule sends in that step; slots a node
 *                                   does not yet hold are never written.
 * A bit copy.  Errors: DPRED_E_INVAL, DPRED_E_ALIGN, DPRED_E_CUDA.
 * Asynchronous on `stream`.
 */
#define DPRED_SCHED_RING 0
#define DPRED_SCHED_BIDIR_RING 1
#define DPRED_SCHED_RECURSIVE_DOUBLING 2
int dpred_allgather_schedule_steps(int32_t schedule, int32_t n_nodes);
int dpred_allgather_schedule_init(int32_t schedule, int32_t n_nodes, int64_t shard_elems, int32_t dtype,
                                  const void* in, void* bufs, void* stream);
int dpred_allgather_schedule_step(int32_t schedule, int32_t n_nodes, int64_t shard_elems, int32_t dtype, void* bufs,
                                  int32_t step, void* stream);

/*
 * Write-only fill (no counterpart in the pages; a measuring aid): writes the
 * 32-bit pattern over bytes of dst (device) and reads nothing, so its rate is
 * the device's HBM write ceiling, the bound of store-dominated kernels such
 * as the AllGather ([AG] "理论下界": its cost is the N·M output).
 *   method 0: 16-byte streaming stores from every thread of a persistent grid
 *             (dst and bytes multiples of 16),
 *   method 1: 32-byte streaming stores (dst and bytes multiples of 32),
 *   method 2: bulk copies (cp.async.bulk) of a 16 KB shared-memory tile by
 *             four issuing warps per CTA (dst and bytes multiples of 16).
 * ctas_per_sm: CTAs per SM of the persistent grid (0 = as many as fit;
 * method 2 takes 0 as 1).  Errors: DPRED_E_INVAL, DPRED_E_ALIGN,
 * DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_fill_pattern(void* dst, size_t bytes, uint32_t pattern, int32_t method, int32_t ctas_per_sm,
                       void* stream);

/*
 * Mixed streaming (no counterpart in the pages; a measuring aid): bulk-loads
 * read_bytes of src (device) into shared memory that nothing reads, and
 * bulk-stores a constant pattern over write_bytes of dst (device), the loads
 * spread evenly between the stores.  No store depends on a load, so the rate
 * is what HBM sustains for this mix of reads and writes -- the ceiling of a
 * kernel with the same mix, e.g. the AllGather (reads M, writes N·M).
 * Buffers and sizes must be multiples of 16 bytes (DPRED_E_ALIGN).  A bounded
 * wait that gives up records DPRED_E_TIMEOUT in the device error word.
 * Errors: DPRED_E_INVAL, DPRED_E_ALIGN, DPRED_E_CUDA.  Asynchronous on `stream`.
 */
int dpred_stream_mixed(const void* src, size_t read_bytes, void* dst, size_t write_bytes, void* stream);

/*
 * Device error word: 0, or the DPRED_E_* code of the first device-side
 * failure (a bounded wait that gave up, an internal consistency check) since
 * the last clear.  Synchronises the current device.  clear != 0 resets it.
 */
int dpred_device_status(int32_t* code, int32_t clear);

/*
 * The device address of page-locked (pinned) host memory, for kernels that
 * read or write host buffers directly over the host link (no counterpart in
 * the pages).  host: any address inside a pinned allocation (cudaHostAlloc,
 * or cudaHostRegister with mapping).  *dev receives the address the current
 * device uses for the same byte; with unified addressing it equals host.
 * Errors: DPRED_E_INVAL (null, or memory that is not pinned and mapped),
 * DPRED_E_CUDA.  Synchronous; enqueues nothing.
 */
int dpred_host_mapped_pointer(const void* host, void** dev);

/*
 * Self-test of the bounded-wait path (no counterpart in the pages): launches
 * one thread that waits on an mbarrier phase nothing completes, gives up after
 * budget_cycles SM clocks (0..4e9) and records DPRED_E_TIMEOUT in the device
 * error word, read back with dpred_device_status.  No fault, no trap: the
 * context stays usable.  Asynchronous on `stream`.
 */
int dpred_selftest_wait_timeout(int64_t budget_cycles, void* stream);

/*
 * Self-test of the bounds-test path (no counterpart in the pages): one thread
 * runs the flush kernels' access test on index 16 of a 16-element range.  The
 * checked build (dpred_checked_build() == 1) records DPRED_E_BOUNDS in the
 * device error word; the default build records nothing.  No memory is
 * accessed in either build.  Asynchronous on `stream`.
 */
int dpred_selftest_bounds(void* stream);

/*
 * Self-test of the flush's pre-division (no counterpart in the pages): for
 * every fp32 bit pattern x (2^32 inputs), and again for every bf16 value,
 * compares the quotient the flush kernels' vector paths use for a rank count
 * of `world` -- a multiply by the exact reciprocal for powers of two; for
 * other counts the division-free forms (Markstein's correction for fp32
 * terms, a split reciprocal for bf16 terms) with IEEE division for the tiny
 * terms their checks flag (no check at the counts where the form is exact on
 * every input) -- with IEEE division x / world rounded to nearest even (two NaNs count as
 * equal).  *mismatches receives the number of differing cases,
 * *first_mismatch the lowest differing bit pattern (0xFFFFFFFF when none).  Runs on the legacy default stream of the current device and
 * synchronises it.  Errors: DPRED_E_INVAL, DPRED_E_CUDA.
 */
int dpred_selftest_prediv(int32_t world, uint64_t* mismatches, uint32_t* first_mismatch);

#ifdef __cplusplus
}
#endif

#endif /* DPRED_H */
