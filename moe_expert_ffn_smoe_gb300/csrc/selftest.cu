// A diagnostic of the bounded device waits the library's kernels use: one
// warp waits for an event that never happens, gives up after the same limit
// the kernels use, records the timeout in the library's status word and
// returns, leaving the context usable.  Nothing is in flight while it waits.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

__device__ unsigned g_never_set = 0;  // no code writes it

__global__ void __launch_bounds__(32) bounded_wait_selftest(int kind, unsigned *status)
{
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    if (kind == 0) {
        // an mbarrier expecting two arrivals that gets one: phase 0 never completes
        const uint32_t b = smem_addr(&bar);
        mbar_init(b, 2);
        fence_mbar_init();
        mbar_arrive(b);
        mbar_wait_bounded(b, 0u, status, 9u);
    } else {
        // a device counter that nothing increments
        if (!wait_count(&g_never_set, 1u)) atomicExch(status, 10u);
    }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int kind, cudaStream_t stream)
{
    unsigned *status = device_status_word();
    if (!status) return cudaErrorInvalidDevice;
    bounded_wait_selftest<<<1, 32, 0, stream>>>(kind, status);
    return cudaGetLastError();
}

}  // namespace smoe
