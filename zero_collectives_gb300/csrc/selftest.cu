// selftest.cu -- exercises the bounded-wait path without any fault: one thread
// waits on an mbarrier phase that nothing will complete, gives up after the
// given clock budget and records DPRED_E_TIMEOUT in the device error word,
// exactly as a real flush wait would.
#include "common.cuh"
#include "tma.cuh"

namespace {

__global__ void wait_timeout_kernel(int* err, long long budget) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        dpred::tma::mbar_init(&bar, 1);  // expects one arrival that never comes
        dpred::tma::fence_barrier_init();
        if (!dpred::tma::mbar_wait(&bar, 0, budget) && err) atomicCAS(err, 0, DPRED_E_TIMEOUT);
    }
}

}  // namespace

extern "C" int dpred_selftest_wait_timeout(int64_t budget_cycles, void* stream) {
    if (budget_cycles < 0 || budget_cycles > 4000000000LL)
        return dpred::set_error(DPRED_E_INVAL, "budget %lld cycles outside 0..4e9", (long long)budget_cycles);
    int* err = dpred::device_error_word();
    if (!err) return dpred::set_error(DPRED_E_CUDA, "device error word unavailable");
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, budget_cycles);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "self-test launch");
}
