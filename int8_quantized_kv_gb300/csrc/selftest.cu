// selftest.cu -- kvq8_selftest_bounded_wait: a check that the library's
// bounded pipeline waits end.  No counterpart on the pages.
//
// Every wait of the decode kernels on a copy or a shared-memory slot is
// bounded: when the bound passes, the kernel ORs KVQ8_DEV_TIMEOUT into the
// caller's status word and unwinds, instead of spinning forever.  A real copy
// that never completes cannot be provoked without faulting the GPU, so this
// entry point runs the same wait routine on an mbarrier phase that nothing
// completes (no thread arrives on it, no copy is issued), which makes the
// bound pass on purpose and nothing else.
#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"
#include "kvq8_ptx.cuh"

namespace kvq8 {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint32_t *dev_status, uint64_t timeout_ns,
                                                                   unsigned long long *waited_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t t0 = global_timer_ns();
    // phase 0 of `bar` completes only when one thread arrives: none does
    const bool completed = mbar_wait_bounded(b, 0, timeout_ns);
    const uint64_t t1 = global_timer_ns();
    if (threadIdx.x == 0) {
        if (!completed) flag_status(dev_status, KVQ8_DEV_TIMEOUT);
        if (waited_ns) *waited_ns = t1 - t0;
    }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint32_t *dev_status, uint64_t timeout_ns, unsigned long long *waited_ns,
                                         cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(dev_status, timeout_ns, waited_ns);
    return cudaGetLastError();
}

}  // namespace kvq8
