// debug_wait.cu -- test hook for the failure path of the bounded waits.
//
// One warp waits on a shared-memory mbarrier that nothing ever arrives at.
// The wait gives up after limit_ns, records CP_ETIMEOUT in the device error
// word and the kernel returns normally: no trap, no fault, the context stays
// usable.  This exercises exactly the wait routine every pipelined kernel of
// the library uses.
#include <cuda_runtime.h>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

__global__ void debug_wait_kernel(unsigned *err, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl wc{err, &abort_flag, limit_ns};
    waitw(smem_u32(&bar), 0, wc);
}

}  // namespace

int launch_debug_wait(unsigned *err, uint64_t limit_ns, cudaStream_t st)
{
    debug_wait_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace cp
