// selftest.cu -- a launch that exercises the library's bounded in-kernel wait:
// one CTA waits on a shared-memory barrier that nothing completes, gives up
// after the given time, flags PD_DEVERR_TIMEOUT and returns, the same way
// every kernel of the library leaves a wait that runs out.  The GPU context
// stays usable afterwards.
#include <cuda_runtime.h>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

__global__ void bounded_wait_selftest_kernel(int32_t* dev_err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);              // one arrival completes the phase; none comes
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_for(&bar, 0, limit_ns)) flag_error(dev_err, PD_DEVERR_TIMEOUT);
}

}  // namespace

pd_status launch_bounded_wait_selftest(int32_t* dev_err, unsigned long long limit_ns,
                                       cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(dev_err, limit_ns);
    return launch_result(cudaGetLastError());
}

}  // namespace pd
