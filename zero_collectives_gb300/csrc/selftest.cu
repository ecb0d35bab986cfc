// selftest.cu -- exercises the device error paths without any fault.
//  * Bounded wait: one thread waits on an mbarrier phase that nothing will
//    complete, gives up after the given clock budget and records
//    DPRED_E_TIMEOUT in the device error word, exactly as a real flush wait
//    would.
//  * Bounds test: one thread runs the flush kernels' access test on an index
//    outside its range.  The checked build records DPRED_E_BOUNDS; the default
//    build compiles the test away.  Nothing is accessed in either build.
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

__global__ void bounds_test_kernel(int* err, int64_t n, int64_t idx) {
    (void)dpred::access_ok(idx >= 0 && idx < n, err);
}

}  // namespace

extern "C" int dpred_selftest_bounds(void* stream) {
    int* err = dpred::device_error_word();
    if (!err) return dpred::set_error(DPRED_E_CUDA, "device error word unavailable");
    bounds_test_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err, 16, 16);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "self-test launch");
}

extern "C" int dpred_selftest_wait_timeout(int64_t budget_cycles, void* stream) {
    if (budget_cycles < 0 || budget_cycles > 4000000000LL)
        return dpred::set_error(DPRED_E_INVAL, "budget %lld cycles outside 0..4e9", (long long)budget_cycles);
    int* err = dpred::device_error_word();
    if (!err) return dpred::set_error(DPRED_E_CUDA, "device error word unavailable");
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, budget_cycles);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DPRED_OK : dpred::cuda_error(e, "self-test launch");
}
