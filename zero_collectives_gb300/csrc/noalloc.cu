// noalloc.cu -- dpred_flush_bucket_noalloc: the bucket flush for callers that
// cannot allocate device memory.
//
// dpred_flush_bucket keeps a large bucket's task table in a device workspace
// that the caller passes in.  Some callers cannot produce one: runtimes that
// hand out all device memory up front from a fixed budget and have nothing
// left to lend, and plug-ins that run inside another framework's allocator
// and may not allocate device memory of their own.  For them this entry point
// uses a fixed scratch array that lives in the library itself instead of a
// caller workspace.
//
// The scratch array is a file-scope __device__ variable, so every GPU that
// loads the library holds its kScratchBytes until the process exits.  Host
// code only sees a stand-in for it; the real device address is looked up
// once per device with cudaGetSymbolAddress (on the first call made on that
// device, with that device current) and passed to the kernel as its
// workspace.  Everything else -- validation, the plan, the kernel -- is the
// unchanged dpred_flush_bucket path.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DPRED_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_flush_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch[kMaxDevices] = {};  // device address of g_flush_scratch, per device ordinal

int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return dpred::cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return dpred::set_error(DPRED_E_INVAL, "device ordinal %d outside 0..%d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_flush_scratch);
        if (e != cudaSuccess || p == nullptr) return dpred::cuda_error(e, "cudaGetSymbolAddress of the flush scratch");
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return DPRED_OK;
}

}  // namespace

extern "C" int dpred_flush_bucket_noalloc(int32_t world, int32_t in_dtype, void* grads, int64_t ld,
                                          const dpred_task* tasks, int32_t n_tasks, const int32_t* owner,
                                          int32_t n_params, int32_t out_dtype, void* const* dst, int32_t pre_div,
                                          int32_t reduce_to_owner, int32_t flags, dpred_probe* probe,
                                          void* stream) {
    if (world < 1 || world > DPRED_MAX_WORLD)
        return dpred::set_error(DPRED_E_INVAL, "world %d outside 1..%d", world, DPRED_MAX_WORLD);
    if (n_tasks < 0) return dpred::set_error(DPRED_E_INVAL, "n_tasks < 0");
    const size_t need = dpred_flush_workspace_bytes(world, n_tasks);
    if (need > kScratchBytes)
        return dpred::set_error(DPRED_E_SIZE,
                                "a bucket of %d tasks at world %d needs %zu bytes of plan scratch; the "
                                "allocation-free flush holds at most %zu (use dpred_flush_bucket with a workspace)",
                                n_tasks, world, need, kScratchBytes);
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != DPRED_OK) return rc;
    return dpred_flush_bucket(world, in_dtype, grads, ld, tasks, n_tasks, owner, n_params, out_dtype, dst, pre_div,
                              reduce_to_owner, flags, probe, scratch, kScratchBytes, stream);
}
