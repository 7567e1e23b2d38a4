// selftest.cu -- the bounded-wait error path, made to fire on purpose.
//
// Every wait of the layer's kernels on an mbarrier is bounded: when it expires the
// kernel records an error bit in the workspace's error word and returns, so that the
// host learns of it through moe_last_device_status and the CUDA context stays usable.
// k_wait_expires runs exactly that path on a barrier no thread ever arrives at (with
// a short limit), which lets a test check the whole chain on a GPU without a stalled
// or faulting kernel.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) k_wait_expires(uint32_t* err, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);  // one arrival expected; none comes
    fence_mbar_init();
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&bar, 0)) {
        if (global_timer_ns() - t0 > timeout_ns) {
            atomicOr(err, kErrTimeoutProducer);
            return;
        }
    }
}

}  // namespace

cudaError_t launch_wait_expires(uint32_t* err, unsigned long long timeout_ns, cudaStream_t st)
{
    return launch_kernel(k_wait_expires, dim3(1), dim3(32), 0, st, false, err, timeout_ns);
}

}  // namespace moe
