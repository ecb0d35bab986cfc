/*
 * datagen.cu -- fill host or device buffers with the seeded values of datagen.h.
 *
 * Element (r, c) of a [rows, cols] matrix (row stride ld elements) is value
 * number (col0 + c) of stream (stream0 + r * stream_step) under `seed`.  The
 * device fill and the host fill call the same datagen.h functions, so they
 * produce the same bits.  Nothing here performs a reduction.
 */
#include <cuda_runtime.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#include "datagen.h"

namespace {

struct FillArgs {
    void* out;
    int dtype, kind;
    int64_t rows, cols, ld, col0;
    uint64_t seed, stream0, stream_step;
    float scale;
};

__host__ __device__ inline void fill_one(const FillArgs& a, int64_t r, int64_t c, uint64_t key) {
    uint64_t i = (uint64_t)(a.col0 + c);
    int64_t off = r * a.ld + c;
    if (a.dtype == DG_BF16) {
        uint16_t v = a.kind == DG_NORMAL ? dg_normal_bf16(key, i, a.scale) : dg_uniform_bf16(key, i);
        ((uint16_t*)a.out)[off] = v;
    } else {
        float v = a.kind == DG_NORMAL ? dg_normal_f32(key, i, a.scale) : dg_uniform_f32(key, i);
        ((float*)a.out)[off] = v;
    }
}

__global__ void fill_kernel(FillArgs a) {
    // One row per blockIdx.y (grid-strided), columns grid-strided along x.
    for (int64_t r = blockIdx.y; r < a.rows; r += gridDim.y) {
        uint64_t key = dg_key(a.seed, a.stream0 + (uint64_t)r * a.stream_step);
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < a.cols;
             c += (int64_t)gridDim.x * blockDim.x)
            fill_one(a, r, c, key);
    }
}

struct HostJob {
    const FillArgs* a;
    int64_t begin, end;  // flat range over rows * cols
};

void* host_worker(void* p) {
    HostJob* j = (HostJob*)p;
    const FillArgs& a = *j->a;
    int64_t e = j->begin;
    while (e < j->end) {
        int64_t r = e / a.cols, c = e % a.cols;
        uint64_t key = dg_key(a.seed, a.stream0 + (uint64_t)r * a.stream_step);
        int64_t stop = (r + 1) * a.cols < j->end ? (r + 1) * a.cols : j->end;
        for (; e < stop; ++e, ++c) fill_one(a, r, c, key);
    }
    return nullptr;
}

bool valid(int dtype, int kind, int64_t rows, int64_t cols, int64_t ld) {
    return (dtype == DG_BF16 || dtype == DG_F32) && (kind == DG_NORMAL || kind == DG_UNIFORM) &&
           rows >= 0 && cols >= 0 && ld >= cols;
}

}  // namespace

extern "C" {

/* sigma * 2^-16 in fp32: the multiplier of the normal recipe. */
float dg_normal_scale(float sigma) { return sigma * (1.0f / 65536.0f); }

int dg_fill_device(void* out, int dtype, int kind, int64_t rows, int64_t cols, int64_t ld, int64_t col0,
                   uint64_t seed, uint64_t stream0, uint64_t stream_step, float scale, void* stream) {
    if (!valid(dtype, kind, rows, cols, ld)) return -1;
    if (rows == 0 || cols == 0) return 0;
    FillArgs a{out, dtype, kind, rows, cols, ld, col0, seed, stream0, stream_step, scale};
    int64_t bx = (cols + 255) / 256;
    if (bx > 4096) bx = 4096;
    int64_t by = rows > 65535 ? 65535 : rows;
    fill_kernel<<<dim3((unsigned)bx, (unsigned)by), 256, 0, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int dg_fill_host(void* out, int dtype, int kind, int64_t rows, int64_t cols, int64_t ld, int64_t col0,
                 uint64_t seed, uint64_t stream0, uint64_t stream_step, float scale, int threads) {
    if (!valid(dtype, kind, rows, cols, ld)) return -1;
    FillArgs a{out, dtype, kind, rows, cols, ld, col0, seed, stream0, stream_step, scale};
    int64_t total = rows * cols;
    if (total == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (total < (int64_t)threads * 65536) threads = 1;
    pthread_t tid[256];
    HostJob jobs[256];
    int64_t per = (total + threads - 1) / threads;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = HostJob{&a, t * per, (t + 1) * per < total ? (t + 1) * per : total};
        if (jobs[t].begin >= jobs[t].end) break;
        if (threads == 1) {
            host_worker(&jobs[t]);
        } else if (pthread_create(&tid[t], nullptr, host_worker, &jobs[t]) == 0) {
            ++started;
        } else {
            host_worker(&jobs[t]);
            tid[t] = 0;
        }
    }
    for (int t = 0; t < threads && threads > 1; ++t)
        if (jobs[t].begin < jobs[t].end && tid[t]) pthread_join(tid[t], nullptr);
    (void)started;
    return 0;
}

/* out[j] = value number idx[j] of stream streams[j]. */
int dg_sample_host(void* out, int dtype, int kind, int64_t count, const uint64_t* streams, const int64_t* idx,
                   uint64_t seed, float scale) {
    if (!valid(dtype, kind, 1, 1, 1) || count < 0) return -1;
    for (int64_t j = 0; j < count; ++j) {
        uint64_t key = dg_key(seed, streams[j]);
        uint64_t i = (uint64_t)idx[j];
        if (dtype == DG_BF16)
            ((uint16_t*)out)[j] = kind == DG_NORMAL ? dg_normal_bf16(key, i, scale) : dg_uniform_bf16(key, i);
        else
            ((float*)out)[j] = kind == DG_NORMAL ? dg_normal_f32(key, i, scale) : dg_uniform_f32(key, i);
    }
    return 0;
}

/* Parameter sizes in [lo, lo + span): sizes[p] = dg_int_range(key(seed, stream), p, lo, span). */
int dg_int_sizes(int64_t* out, int64_t count, uint64_t seed, uint64_t stream, int64_t lo, int64_t span) {
    if (count < 0 || span <= 0) return -1;
    uint64_t key = dg_key(seed, stream);
    for (int64_t p = 0; p < count; ++p) out[p] = dg_int_range(key, (uint64_t)p, lo, span);
    return 0;
}

}  // extern "C"
