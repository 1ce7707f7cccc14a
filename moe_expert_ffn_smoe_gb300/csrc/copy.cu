// Copies between any two device-accessible buffers (device memory, or pinned
// host memory, which on a Grace-Blackwell node the SMs reach over the
// coherent chip-to-chip link), done by the SMs rather than a copy engine:
// a token's input and its outputs move between host and device inside the
// same chain of kernels as the step, with programmatic dependent launch on
// both sides.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

constexpr int COPY_THREADS = 256;

__global__ void __launch_bounds__(COPY_THREADS) copy16(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                      size_t n)
{
    // dst may be read by the kernel before this one: wait for it to finish
    pdl_wait();
    const size_t stride = static_cast<size_t>(gridDim.x) * COPY_THREADS;
    for (size_t i = static_cast<size_t>(blockIdx.x) * COPY_THREADS + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_copy16(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const size_t n = bytes / 16;
    // about 4 uint4 per thread, at most one CTA per SM
    size_t blocks = (n + 4 * COPY_THREADS - 1) / (4 * COPY_THREADS);
    if (blocks < 1) blocks = 1;
    if (blocks > static_cast<size_t>(dev->sm_count)) blocks = static_cast<size_t>(dev->sm_count);
    return launch_pdl(copy16, dim3(static_cast<unsigned>(blocks)), dim3(COPY_THREADS), 0, stream,
                      static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n);
}

// Device address of a buffer the device can access, or null: device and
// managed memory as they are, pinned (page-locked, registered) host memory
// through its mapped device address.
void *device_address(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        return const_cast<void *>(p);
    case cudaMemoryTypeHost:
        return at.devicePointer;
    default:
        return nullptr;  // pageable host memory
    }
}

}  // namespace smoe
