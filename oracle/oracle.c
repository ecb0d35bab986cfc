/*
 * oracle.c -- plain, slow CPU oracle of the ZeRO-1 gradient-reduction path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  The CUDA library never
 * calls it and shares no code with it.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -shared -fPIC.  Every
 * floating-point step below is one IEEE fp32 operation in round-to-nearest
 * mode, in the order written; contraction into FMA is disabled so no two
 * steps fuse.
 *
 * Sources (pages):
 *  [DS]  DeepSpeed issue #8700, "[REQUEST] DeepCompile ZeRO-1: reduce-to-owner
 *        instead of AllReduce".
 *  [MT]  MaxText PR #5099, "Defer the data-parallel gradient all-reduce to
 *        update() under gradient accumulation".
 *  [AG]  "AllGather" (tier6-model interconnect notes, 集合通信 / all-gather).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes):
 *  - The partition size of a group of T elements over S ranks is ceil(T/S);
 *    partitions are contiguous in the group's flat (model) order, no padding.
 *  - The reduction is an fp32 sum in rank order 0..W-1 that starts from the
 *    rank-0 term (not from 0.0, so -0 survives); pre-division is an fp32
 *    IEEE division of each upcast term by W; the result is rounded once to
 *    the output type (bf16: round to nearest, ties to even).
 *  - A parameter of a group whose communicator is not the data-parallel one
 *    has no owner and every data-parallel rank is treated as holding it.
 *  - A zero-element parameter has no owner and no holders.
 *
 * Parity: every function here is pinned by the tests under tests/ (closed
 * forms, the worked tables of [AG], the probe line of [DS], brute force and
 * exactness cases); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_F32 1

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the upper half of an IEEE binary32 pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to bf16, round-to-nearest, ties-to-even, written out
 * from the definition: keep the upper 16 bits, look at the 16 dropped bits;
 * above half -> round up, below -> down, exactly half -> make the kept part
 * even.  NaN stays NaN (quiet bit set); infinities and overflow to infinity
 * follow from the same carry into the exponent. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

static float load_elem(int dt, const void* base, int64_t i) {
    if (dt == ORC_BF16) return orc_bf16_to_f32(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

static void store_elem(int dt, void* base, int64_t i, float v) {
    if (dt == ORC_BF16)
        ((uint16_t*)base)[i] = orc_f32_to_bf16(v);
    else
        ((float*)base)[i] = v;
}

static int dtype_ok(int dt) { return dt == ORC_BF16 || dt == ORC_F32; }

/* ------------------------------------------------------- element reduce --- */

/* One reduced element: [DS] "Describe the solution you'd like" -- the same
 * reduction with the same operand order per element as the AllReduce it
 * replaces; design point "Summation semantics untouched" -- pre-division by
 * the world size before the sum (pre_div), then the sum (ncclSum). */
static float reduce_one(int world, int in_dt, const void* x, int64_t ld, int64_t k, int pre_div) {
    float wf = (float)world;
    float y = 0.0f;
    for (int r = 0; r < world; ++r) {
        float t = load_elem(in_dt, x, (int64_t)r * ld + k);
        if (pre_div) t = t / wf;
        if (r == 0)
            y = t;
        else
            y = y + t;
    }
    return y;
}

/* out[k] = reduced element k of rows x[0..world-1] (row stride ld), k < m. */
int orc_reduce_rows(int world, int in_dt, const void* x, int64_t ld, int64_t m, int pre_div, int out_dt,
                    void* out) {
    if (world < 1 || !dtype_ok(in_dt) || !dtype_ok(out_dt) || m < 0 || ld < m) return -1;
    for (int64_t k = 0; k < m; ++k) store_elem(out_dt, out, k, reduce_one(world, in_dt, x, ld, k, pre_div));
    return 0;
}

/* ------------------------------------------------------------ owner map --- */

/* [DS] "Design points":
 *  - "Owner map costs nothing to build": param_to_partition_ids lists every
 *    partition holding a piece of the parameter; exactly one entry means
 *    exactly one owner, that entry's rank.  The map depends on nothing
 *    rank-specific, so `rank` is accepted and ignored.
 *  - "Partial parameters keep AllReduce": two or more entries -> not declared
 *    (owner -1).
 *  - "Parameter groups reduced over a different communicator are skipped":
 *    eligible iff the group's size equals the world size and its group rank
 *    i maps to global rank i for every i.
 *  - "No native flag": with reduce_to_owner off no owner is declared.
 * Holders (ranks with a real gradient buffer, [DS] "Is your feature request
 * related to a problem?") are the ranks in the parameter's partition list.
 *
 * Groups are passed flattened: group g has comm_size[g] ranks listed in
 * comm_ranks (concatenated) and n_params[g] sizes in numel (concatenated).
 * Outputs are per parameter, in concatenated order. */
int orc_owner_map(int world, int rank, int n_groups, const int32_t* comm_size, const int32_t* comm_ranks,
                  const int32_t* n_params, const int64_t* numel, int reduce_to_owner, int32_t* owner,
                  int32_t* holder_lo, int32_t* holder_hi, int32_t* n_owned, int32_t* n_total) {
    (void)rank;
    if (world < 1 || n_groups < 0) return -1;
    int64_t pbase = 0, rbase = 0;
    int32_t owned = 0, total = 0;
    for (int g = 0; g < n_groups; ++g) {
        int S = comm_size[g];
        if (S < 1 || n_params[g] < 0) return -1;
        int eligible = (S == world);
        for (int i = 0; i < S && eligible; ++i)
            if (comm_ranks[rbase + i] != i) eligible = 0;
        int64_t T = 0;
        for (int p = 0; p < n_params[g]; ++p) {
            if (numel[pbase + p] < 0) return -1;
            T += numel[pbase + p];
        }
        int64_t P = (T + S - 1) / S; /* partition size */
        int64_t s = 0;
        for (int p = 0; p < n_params[g]; ++p) {
            int64_t n = numel[pbase + p];
            int64_t e = s + n;
            /* param_to_partition_ids: every partition j whose range
             * [j*P, (j+1)*P) intersects [s, e). */
            int entries = 0, first = -1, last = -1;
            for (int j = 0; j < S && n > 0; ++j) {
                int64_t lo = (int64_t)j * P, hi = (int64_t)(j + 1) * P;
                if (hi > T) hi = T;
                if (lo < e && s < hi) {
                    if (entries == 0) first = j;
                    last = j;
                    ++entries;
                }
            }
            int64_t out = pbase + p;
            if (n == 0) {
                owner[out] = -1;
                holder_lo[out] = -1;
                holder_hi[out] = -1;
            } else if (!eligible) {
                owner[out] = -1;
                holder_lo[out] = 0;
                holder_hi[out] = world - 1;
            } else {
                owner[out] = (reduce_to_owner && entries == 1) ? first : -1;
                holder_lo[out] = first;
                holder_hi[out] = last;
            }
            if (owner[out] >= 0) ++owned;
            ++total;
            s = e;
        }
        pbase += n_params[g];
        rbase += S;
    }
    *n_owned = owned;
    *n_total = total;
    return 0;
}

/* --------------------------------------------------------- bucket flush --- */

/* Probe counters of one flush from its metadata alone ([DS] "reduce_probe":
 * reduced_elems, kept_elems, discarded and how much took the owner path).
 * has_dst[r * n_tasks + t] != 0 when rank r has a real buffer for task t;
 * has_dst == NULL means the in-place form, where a rank keeps what is
 * delivered to its row.  probe[0] = tasks, [1] = reduced_elems (sum of task
 * sizes), [2] = owner_tasks, [3] = owner_elems, [4 + r] = kept_elems[r]. */
int orc_flush_probe(int world, int n_tasks, const int32_t* task_param, const int64_t* task_numel,
                    const int32_t* owner, int n_params, const uint8_t* has_dst, int reduce_to_owner,
                    int64_t* probe) {
    if (world < 1 || n_tasks < 0) return -1;
    probe[0] = n_tasks;
    probe[1] = probe[2] = probe[3] = 0;
    for (int r = 0; r < world; ++r) probe[4 + r] = 0;
    for (int t = 0; t < n_tasks; ++t) {
        if (owner != NULL && (task_param[t] < 0 || task_param[t] >= n_params)) return -1;
        int root = (reduce_to_owner && owner != NULL && owner[task_param[t]] >= 0) ? owner[task_param[t]] : -1;
        probe[1] += task_numel[t];
        if (root >= 0) {
            probe[2] += 1;
            probe[3] += task_numel[t];
        }
        for (int r = 0; r < world; ++r) {
            int kept = has_dst ? has_dst[(int64_t)r * n_tasks + t] != 0 : (root < 0 || root == r);
            if (kept) probe[4 + r] += task_numel[t];
        }
    }
    return 0;
}

/* The ZeRO-1 bucket flush, [DS]:
 *  1. roots: for every task, root = owner of its parameter when the
 *     reduce-to-owner path is on and the parameter has an owner, else -1
 *     ("roots is therefore precomputed for the whole bucket").
 *  2. reduce every element (pre-division, then the rank-order sum).
 *  3. deliver: root >= 0 -> only rank root (ncclReduce(root=owner)); root -1
 *     -> every rank (ncclAllReduce).
 *  4. copy-out: a delivered rank whose buffer is empty is skipped ("if
 *     (grad_buf.numel() == 0) { continue; }").  dst[r * n_tasks + t] is rank
 *     r's buffer for task t, NULL for an empty one.  With dst == NULL the
 *     result is written in place into the delivered ranks' bucket rows
 *     (grads row r, the task's range); out_dt must then equal in_dt.
 *  5. probe: the counters of orc_flush_probe, when probe != NULL.
 * grads is [world, ld]; task t covers [task_off[t], task_off[t] + task_numel[t])
 * of every row.  owner is indexed by parameter id and may be NULL (no owners). */
int orc_flush(int world, int in_dt, void* grads, int64_t ld, int n_tasks, const int32_t* task_param,
              const int64_t* task_off, const int64_t* task_numel, const int32_t* owner, int n_params,
              int out_dt, void* const* dst, int pre_div, int reduce_to_owner, int64_t* probe) {
    if (world < 1 || !dtype_ok(in_dt) || !dtype_ok(out_dt) || n_tasks < 0) return -1;
    if (dst == NULL && out_dt != in_dt) return -1;
    for (int t = 0; t < n_tasks; ++t) {
        if (task_off[t] < 0 || task_numel[t] < 0 || task_off[t] + task_numel[t] > ld) return -1;
        if (owner != NULL && (task_param[t] < 0 || task_param[t] >= n_params)) return -1;
    }
    int* root = (int*)malloc(sizeof(int) * (size_t)(n_tasks > 0 ? n_tasks : 1));
    if (!root) return -1;
    for (int t = 0; t < n_tasks; ++t)
        root[t] = (reduce_to_owner && owner != NULL && owner[task_param[t]] >= 0) ? owner[task_param[t]] : -1;

    for (int t = 0; t < n_tasks; ++t) {
        for (int64_t k = 0; k < task_numel[t]; ++k) {
            int64_t col = task_off[t] + k;
            float y = reduce_one(world, in_dt, grads, ld, col, pre_div);
            for (int r = 0; r < world; ++r) {
                int delivered = (root[t] < 0) || (root[t] == r);
                if (!delivered) continue;
                if (dst == NULL) {
                    store_elem(out_dt, grads, (int64_t)r * ld + col, y);
                } else {
                    void* d = dst[(int64_t)r * n_tasks + t];
                    if (d == NULL) continue; /* empty buffer: skipped in copy-out */
                    store_elem(out_dt, d, k, y);
                }
            }
        }
    }
    free(root);
    if (probe) {
        uint8_t* has = NULL;
        if (dst != NULL) {
            has = (uint8_t*)malloc((size_t)world * (size_t)(n_tasks > 0 ? n_tasks : 1));
            if (!has) return -1;
            for (int64_t i = 0; i < (int64_t)world * n_tasks; ++i) has[i] = dst[i] != NULL;
        }
        int rc = orc_flush_probe(world, n_tasks, task_param, task_numel, owner, n_params, has, reduce_to_owner, probe);
        free(has);
        return rc;
    }
    return 0;
}

/* ------------------------------------------------ deferred accumulation --- */

/* [MT] "What": per-replica partial sums accumulate replica-locally across
 * micro-batches; update() then performs the single cross-replica all-reduce.
 * acc and g are [world, n] (contiguous rows).  For every replica r and k:
 *   a = first ? g[r][k] : acc[r][k] + g[r][k]         (fp32)
 * finalize == 0: acc[r][k] = a.
 * finalize == 1: total[k] = (a[0] + a[1] + ... + a[world-1]) * scale, the sum
 * in rank order from the rank-0 term; acc is left unchanged (the accumulator
 * is consumed by the reduction, which "update() reshards back to a plain
 * spec" performs once).  scale is a caller factor such as 1/denominator
 * ([MT] "_accumulated_denominator is deliberately left plain"). */
int orc_accumulate(int world, int64_t n, float* acc, int g_dt, const void* g, int first, int finalize, float scale,
                   float* total) {
    if (world < 1 || n < 0 || !dtype_ok(g_dt)) return -1;
    if (finalize && total == NULL) return -1;
    if (!finalize) {
        for (int r = 0; r < world; ++r)
            for (int64_t k = 0; k < n; ++k) {
                int64_t i = (int64_t)r * n + k;
                float gv = load_elem(g_dt, g, i);
                acc[i] = first ? gv : acc[i] + gv;
            }
        return 0;
    }
    for (int64_t k = 0; k < n; ++k) {
        float y = 0.0f;
        for (int r = 0; r < world; ++r) {
            int64_t i = (int64_t)r * n + k;
            float gv = load_elem(g_dt, g, i);
            float a = first ? gv : acc[i] + gv;
            if (r == 0)
                y = a;
            else
                y = y + a;
        }
        total[k] = y * scale;
    }
    return 0;
}

/* The status quo of [MT] "What": the gradient is all-reduced across
 * replicas once per micro-batch and the reduced micro-batch sums are then
 * accumulated.  g is [n_mb][world][n]; out[k] = (sum over m in order of
 * (sum over r in order of g[m][r][k])) * scale. */
int orc_reduce_each_microbatch(int world, int n_mb, int64_t n, int g_dt, const void* g, float scale, float* out) {
    if (world < 1 || n_mb < 1 || n < 0 || !dtype_ok(g_dt)) return -1;
    for (int64_t k = 0; k < n; ++k) {
        float acc = 0.0f;
        for (int m = 0; m < n_mb; ++m) {
            float s = 0.0f;
            for (int r = 0; r < world; ++r) {
                float v = load_elem(g_dt, g, ((int64_t)m * world + r) * n + k);
                s = (r == 0) ? v : s + v;
            }
            acc = (m == 0) ? s : acc + s;
        }
        out[k] = acc * scale;
    }
    return 0;
}

/* --------------------------------------------- ReduceScatter, AllGather --- */

/* [AG] "与 ReduceScatter 的对偶关系" (duality table): ReduceScatter takes M
 * elements per node and leaves node i with the reduced shard i of M/N
 * elements.  in is [N, M]; out is [N, M/N]; out[i][k] is the reduction (same
 * element rule as the flush) of in[0..N-1][i*S + k].  M % N != 0 -> -3. */
int orc_reduce_scatter(int n_nodes, int64_t m_elems, int in_dt, const void* in, int out_dt, void* out, int pre_div) {
    if (n_nodes < 1 || m_elems < 0 || !dtype_ok(in_dt) || !dtype_ok(out_dt)) return -1;
    if (m_elems % n_nodes != 0) return -3;
    int64_t S = m_elems / n_nodes;
    for (int i = 0; i < n_nodes; ++i)
        for (int64_t k = 0; k < S; ++k)
            store_elem(out_dt, out, (int64_t)i * S + k, reduce_one(n_nodes, in_dt, in, m_elems, i * S + k, pre_div));
    return 0;
}

/* [AG] "语义定义", eq. ag-semantic-output: node i ends with
 * B_i = [A_0, ..., A_{N-1}] (order 0).  [AG] "Ring AllGather", N=4 table:
 * after the ring schedule node i holds [A_i, A_{i-1}, ..., A_{i-N+1}]
 * (indices mod N; order 1), which orc_ring_allgather_steps derives step by
 * step.  in is [N, S] (node j's shard A_j), out is [N, N*S]; a byte copy. */
int orc_allgather(int n_nodes, int64_t shard_elems, int esize, const void* in, void* out, int order) {
    if (n_nodes < 1 || shard_elems < 0 || esize < 1 || (order != 0 && order != 1)) return -1;
    size_t bytes = (size_t)shard_elems * (size_t)esize;
    for (int i = 0; i < n_nodes; ++i)
        for (int c = 0; c < n_nodes; ++c) {
            int src = (order == 0) ? c : ((i - c) % n_nodes + n_nodes) % n_nodes;
            memcpy((char*)out + ((size_t)i * n_nodes + c) * bytes, (const char*)in + (size_t)src * bytes, bytes);
        }
    return 0;
}

/* [AG] "Ring AllGather": N-1 steps; in each step every node forwards the
 * chunk it received in the previous step (its own chunk in step 1) to its
 * right neighbour and receives one chunk from its left neighbour, appending
 * it to its list.  Direction: data moves from node i to node i+1 (the table
 * shows Node 0 receiving D from Node 3 in step 1).
 * hold is [N][N][N]: hold[s][i][c] = chunk id at position c of node i's list
 * after step s (s = 0 is the initial state), -1 where the list is shorter.
 * recv[i] = chunks node i received. */
int orc_ring_allgather_steps(int n, int32_t* hold, int64_t* recv) {
    if (n < 1 || n > 64) return -1;
    int32_t last[64], incoming[64], len[64];
    for (int i = 0; i < n * n * n; ++i) hold[i] = -1;
    for (int i = 0; i < n; ++i) {
        hold[(0 * n + i) * n + 0] = i;
        last[i] = i;
        len[i] = 1;
        recv[i] = 0;
    }
    for (int s = 1; s < n; ++s) {
        for (int i = 0; i < n; ++i) incoming[(i + 1) % n] = last[i]; /* send right */
        for (int i = 0; i < n; ++i) {
            for (int c = 0; c < len[i]; ++c) hold[(s * n + i) * n + c] = hold[((s - 1) * n + i) * n + c];
            hold[(s * n + i) * n + len[i]] = incoming[i];
            len[i] += 1;
            last[i] = incoming[i];
            recv[i] += 1;
        }
    }
    return 0;
}

/* [AG] "Recursive Doubling AllGather": for N = 2^k nodes, log2 N steps; in
 * step j (j = 1..log2 N) node i exchanges everything it holds with the node
 * at distance 2^(j-1).  Simulated with chunk sets.
 * partner is [log2N][N]; xfer[j-1] = chunks each node sends in step j;
 * held[j-1] = chunks each node holds after step j; final_hold is [N][N]:
 * final_hold[i][c] = chunk stored at position c of node i's buffer (received
 * blocks are stored at their own index).  recv[i] = chunks node i received.
 * Returns -1 unless N is a power of two (the page: "适合 N = 2^k 节点"). */
int orc_rd_allgather_steps(int n, int32_t* partner, int64_t* xfer, int64_t* held, int32_t* final_hold, int64_t* recv) {
    if (n < 1 || n > 64 || (n & (n - 1)) != 0) return -1;
    uint64_t have[64], next[64];
    int steps = 0;
    while ((1 << steps) < n) ++steps;
    for (int i = 0; i < n; ++i) {
        have[i] = 1ull << i;
        recv[i] = 0;
    }
    for (int j = 1; j <= steps; ++j) {
        int dist = 1 << (j - 1);
        int64_t sent = -1;
        for (int i = 0; i < n; ++i) {
            int p = i ^ dist;
            partner[(j - 1) * n + i] = p;
            int64_t cnt = 0;
            for (int c = 0; c < n; ++c) cnt += (have[p] >> c) & 1ull;
            if (sent < 0) sent = cnt;
            if (cnt != sent) return -2; /* volumes must be equal across nodes */
            next[i] = have[i] | have[p];
            recv[i] += cnt;
        }
        xfer[j - 1] = sent;
        for (int i = 0; i < n; ++i) have[i] = next[i];
        int64_t h = 0;
        for (int c = 0; c < n; ++c) h += (have[0] >> c) & 1ull;
        held[j - 1] = h;
    }
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < n; ++c) final_hold[i * n + c] = ((have[i] >> c) & 1ull) ? c : -1;
    return 0;
}

/* ------------------------------------------------------ array helpers --- */

/* Element-wise bf16 <-> f32 over arrays (the scalar rules above). */
void orc_bf16_to_f32_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}

void orc_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

/* --------------------------------------------- accumulator checkpoints --- */

/* [MT] "What else had to change", "Accumulator lifetime": a checkpoint holds
 * the reduced total, so saving runs the pending cross-replica all-reduce:
 * total[k] = acc[0][k] + acc[1][k] + ... + acc[W-1][k] (rank order, fp32,
 * from the rank-0 term).  acc is [world, n]; nothing is scaled. */
int orc_accumulator_save(int world, int64_t n, const float* acc, float* total) {
    if (world < 1 || n < 0) return -1;
    for (int64_t k = 0; k < n; ++k) {
        float y = 0.0f;
        for (int r = 0; r < world; ++r) y = (r == 0) ? acc[k] : y + acc[(int64_t)r * n + k];
        total[k] = y;
    }
    return 0;
}

/* Same section: moving a reduced value back onto the unreduced form leaves
 * the value on one replica and zeros on the rest, so the deferred all-reduce
 * reproduces it: acc[0][k] = total[k], acc[r][k] = +0 for r > 0. */
int orc_accumulator_restore(int world, int64_t n, float* acc, const float* total) {
    if (world < 1 || n < 0) return -1;
    for (int64_t k = 0; k < n; ++k) acc[k] = total[k];
    for (int r = 1; r < world; ++r)
        for (int64_t k = 0; k < n; ++k) acc[(int64_t)r * n + k] = 0.0f;
    return 0;
}

/* ------------------------------------- partitioned (ReduceScatter) flush --- */

/* [DS] "Describe alternatives you've considered", ncclReduceScatter over the
 * bucket ("the better end state"), and "Follow-up" (ZeRO-2 registers real
 * buffers with offsets): every rank receives exactly the part of the reduced
 * bucket that lies in its optimizer partition.  Element k of task t belongs
 * to flat position f = flat_offset[param] + k of its group; it goes to rank
 * r = f / part_size at position f - r * part_size of that rank's partition
 * buffer part_dst[r] (NULL: the rank receives nothing).  The value is the
 * same element reduction as the flush.  probe (may be NULL): [0] tasks,
 * [1] reduced_elems, [2] tasks lying inside one partition, [3] their
 * elements, [4 + r] elements delivered to rank r. */
int orc_flush_partitioned(int world, int in_dt, const void* grads, int64_t ld, int n_tasks, const int32_t* task_param,
                          const int64_t* task_off, const int64_t* task_numel, const int64_t* flat_offset,
                          int64_t part_size, int out_dt, void* const* part_dst, int pre_div, int64_t* probe) {
    if (world < 1 || !dtype_ok(in_dt) || !dtype_ok(out_dt) || n_tasks < 0 || part_size < 1) return -1;
    for (int t = 0; t < n_tasks; ++t) {
        if (task_off[t] < 0 || task_numel[t] < 0 || task_off[t] + task_numel[t] > ld) return -1;
        int64_t s = flat_offset[task_param[t]];
        if (s < 0 || (task_numel[t] > 0 && (s + task_numel[t] - 1) / part_size >= world)) return -1;
    }
    if (probe) {
        probe[0] = n_tasks;
        probe[1] = probe[2] = probe[3] = 0;
        for (int r = 0; r < world; ++r) probe[4 + r] = 0;
    }
    for (int t = 0; t < n_tasks; ++t) {
        const int64_t s = flat_offset[task_param[t]];
        for (int64_t k = 0; k < task_numel[t]; ++k) {
            const int64_t f = s + k;
            const int r = (int)(f / part_size);
            const float y = reduce_one(world, in_dt, grads, ld, task_off[t] + k, pre_div);
            if (part_dst[r] != NULL) {
                store_elem(out_dt, part_dst[r], f - (int64_t)r * part_size, y);
                if (probe) probe[4 + r] += 1;
            }
        }
        if (probe) {
            probe[1] += task_numel[t];
            if (task_numel[t] > 0 && s / part_size == (s + task_numel[t] - 1) / part_size) {
                probe[2] += 1;
                probe[3] += task_numel[t];
            }
        }
    }
    return 0;
}

/* The relayout pass of [DS] "Describe alternatives you've considered": the
 * bucket, in gradient-arrival order, is rewritten so that every replica row
 * holds the elements bound for rank 0, then those for rank 1, ..., each
 * rank's run in flat order and padded to `seg` elements: out[q][r * seg + j]
 * is the j-th element (in flat order) of the bucket that lies in partition r,
 * taken from replica row q.  ReduceScatter of out over the W rows then
 * delivers to rank r the reduced run r.  seg_used[r] receives the run
 * lengths; elements past them are not written.  A plain copy. */
int orc_bucket_relayout(int world, int esize, const void* grads, int64_t ld, int n_tasks, const int32_t* task_param,
                        const int64_t* task_off, const int64_t* task_numel, const int64_t* flat_offset,
                        int64_t part_size, int64_t seg, void* out, int64_t out_ld, int64_t* seg_used) {
    if (world < 1 || esize < 1 || n_tasks < 0 || part_size < 1 || seg < 0) return -1;
    /* run start of every rank = smallest flat position of the bucket in that partition */
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * (size_t)world);
    if (!first) return -1;
    for (int r = 0; r < world; ++r) {
        first[r] = -1;
        seg_used[r] = 0;
    }
    for (int t = 0; t < n_tasks; ++t) {
        const int64_t s = flat_offset[task_param[t]];
        for (int64_t k = 0; k < task_numel[t]; ++k) {
            const int64_t f = s + k;
            const int r = (int)(f / part_size);
            if (r >= world) { free(first); return -1; }
            if (first[r] < 0 || f < first[r]) first[r] = f;
            seg_used[r] += 1;
        }
    }
    for (int r = 0; r < world; ++r)
        if (seg_used[r] > seg) { free(first); return -3; }
    /* the bucket's elements in one partition must be one contiguous flat run */
    for (int t = 0; t < n_tasks; ++t) {
        const int64_t s = flat_offset[task_param[t]];
        for (int64_t k = 0; k < task_numel[t]; ++k) {
            const int64_t f = s + k;
            const int r = (int)(f / part_size);
            const int64_t j = f - first[r];
            if (j >= seg_used[r]) { free(first); return -1; }
            for (int q = 0; q < world; ++q)
                memcpy((char*)out + ((int64_t)q * out_ld + (int64_t)r * seg + j) * esize,
                       (const char*)grads + ((int64_t)q * ld + task_off[t] + k) * esize, (size_t)esize);
        }
    }
    free(first);
    return 0;
}

/* [AG] "Ring AllGather", the bidirectional ring (eq. ag-bidir-ring): data
 * moves both ways round the ring at once, so ceil((N-1)/2) steps suffice.  In
 * step s node i receives chunk (i - s) mod N from its left neighbour and chunk
 * (i + s) mod N from its right neighbour (the same chunk once when they
 * coincide).  Chunks are kept at their own index (canonical placement).
 * hold is [steps + 1][N][N]: hold[s][i][c] = c when node i holds chunk c after
 * step s, else -1.  recv[i] = chunks node i received.  Returns the number of
 * steps, or -1. */
int orc_bidir_ring_allgather_steps(int n, int32_t* hold, int64_t* recv) {
    if (n < 1 || n > 64) return -1;
    int steps = n / 2;            /* ceil((n - 1) / 2) */
    uint64_t have[64];
    for (int i = 0; i < n; ++i) {
        have[i] = 1ull << i;
        recv[i] = 0;
    }
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < n; ++c) hold[(0 * n + i) * n + c] = ((have[i] >> c) & 1ull) ? c : -1;
    for (int s = 1; s <= steps; ++s) {
        uint64_t next[64];
        for (int i = 0; i < n; ++i) {
            int from_left = ((i - s) % n + n) % n, from_right = (i + s) % n;
            uint64_t add = (1ull << from_left) | (1ull << from_right);
            /* the chunk from the left must be held by the left neighbour, the chunk from the right by the right one */
            if (!((have[(i - 1 + n) % n] >> from_left) & 1ull) || !((have[(i + 1) % n] >> from_right) & 1ull)) return -2;
            uint64_t fresh = add & ~have[i];
            for (int c = 0; c < n; ++c) recv[i] += (fresh >> c) & 1ull;
            next[i] = have[i] | add;
        }
        for (int i = 0; i < n; ++i) have[i] = next[i];
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < n; ++c) hold[((int64_t)s * n + i) * n + c] = ((have[i] >> c) & 1ull) ? c : -1;
    }
    return steps;
}
