// selftest.cu -- a diagnostic kernel for the device-side failure detection:
// it makes the bounded mbarrier waits of the hot-path kernels run out, with
// no fault and no hang. Two waits on mbarriers that nothing ever completes:
//   warp 0 waits with a short limit, gives up, sets the CTA's abort flag and
//          the device status word (GLA_ERR_TIMEOUT at the next gla_check);
//   warp 1 waits with the kernels' full limit (2 s) and must leave as soon as
//          it sees the abort flag.
// result[0], result[1]: 1 if the wait completed, 0 if it gave up;
// result[2]: microseconds warp 1 waited.
#include <limits.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace gla {
namespace {

using namespace ptx;

__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned int *status, uint64_t limit_ns, int *result) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_word;
    volatile int *abort_flag = &abort_word;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{abort_flag, status};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0 && lane == 0) {
        result[0] = mbar_wait_for(smem_u32(&bars[0]), 0, ctl, limit_ns) ? 1 : 0;
    } else if (warp == 1 && lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        result[1] = mbar_wait(smem_u32(&bars[1]), 0, ctl) ? 1 : 0;
        const uint64_t us = (globaltimer_ns() - t0) / 1000;
        result[2] = us > (uint64_t)INT_MAX ? INT_MAX : (int)us;
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int *status, uint64_t limit_ns, int *result, cudaStream_t s,
                                 int *launches) {
    wait_timeout_kernel<<<1, 64, 0, s>>>(status, limit_ns, result);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
