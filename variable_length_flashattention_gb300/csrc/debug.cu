// debug.cu -- test hook for the bounded waits every kernel of this library
// uses: one CTA waits on an mbarrier that nothing arrives on, gives up after
// the wait limit like any pipeline wait, and reports VFA_ERR_TIMEOUT through
// the status word, leaving the context usable.
#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

__global__ void __launch_bounds__(64) bounded_wait_kernel(int32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&bar), 1);       // one arrival expected; none will come
        fence_barrier_init();
    }
    __syncthreads();
    volatile int *abort = &s_abort;
    const bool done = mbar_wait(smem_u32(&bar), 0, abort);
    __syncthreads();
    if (threadIdx.x == 0 && (!done || *abort) && status)
        atomicCAS(status, 0, VFA_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_debug_bounded_wait(int32_t *status, cudaStream_t stream)
{
    bounded_wait_kernel<<<1, 64, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace vfa
