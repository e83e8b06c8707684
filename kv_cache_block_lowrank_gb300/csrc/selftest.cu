// selftest.cu -- failure-detection self-test: a pipeline wait that runs out.
//
// Every mbarrier wait in the tcgen05 kernels gives up after a time limit, reports
// HSS_ERR_DEVICE_TIMEOUT and lets the kernel exit, so a stalled pipeline ends as an error
// the host can read instead of a hung GPU.  This kernel exercises that path on purpose: one
// thread waits, with the same bounded wait, on a barrier that nothing ever arrives on.
#include "ptx.cuh"

namespace hss {
namespace {

__global__ void wait_timeout_kernel(int32_t* dev_status, int32_t* lib_error, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Phase 0 of `bar` never completes: nobody arrives.
        if (!mbar_wait_for(&bar, 0, limit_ns))
            raise_error(dev_status, lib_error, HSS_ERR_DEVICE_TIMEOUT);
    }
}

}  // namespace
}  // namespace hss

using namespace hss;

extern "C" hss_status hss_self_test_wait_timeout(int32_t* dev_status, int64_t limit_ns,
                                                 void* stream) {
    if (dev_status == nullptr) return HSS_ERR_NULL_POINTER;
    if (limit_ns < 1000 || limit_ns > 2000000000) return HSS_ERR_INVALID_ARGUMENT;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        dev_status, dev->error_word, static_cast<uint64_t>(limit_ns));
    return cudaGetLastError() == cudaSuccess ? HSS_OK : HSS_ERR_CUDA;
}
