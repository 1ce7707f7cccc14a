// Device helpers shared by the sm_103a kernels of libsmoe.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smoe {

constexpr unsigned FULL_MASK = 0xffffffffu;

// 16-byte streaming load of read-only data (weights): non-coherent path,
// no L1 allocation (every weight byte is read exactly once per call).
__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float ldg_f32(const float *p)
{
    float v;
    asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  `pdl_wait` blocks until every grid this
// one depends on has completed and its memory is visible (it returns at
// once for a grid launched without the attribute); `pdl_launch_dependents`
// lets the next grid in the stream start launching.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bulk L2 prefetch of [p, p + bytes): p 16-byte aligned, bytes a multiple of
// 16.  A prefetch only warms L2 (the device-wide point of coherence), so it
// is safe to issue before pdl_wait.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetches the 16-byte-aligned interior of [begin, begin + bytes) into L2,
// split into pieces of at most `piece` bytes spread over the threads of the
// block.  Rounding inward keeps every prefetched byte inside the range.
__device__ __forceinline__ void prefetch_range_l2(const void *begin, size_t bytes, uint32_t piece)
{
    uintptr_t b = reinterpret_cast<uintptr_t>(begin);
    uintptr_t e = b + bytes;
    uintptr_t b16 = (b + 15) & ~uintptr_t(15);
    uintptr_t e16 = e & ~uintptr_t(15);
    if (e16 <= b16) return;
    size_t n = e16 - b16;
    size_t npieces = (n + piece - 1) / piece;
    for (size_t i = threadIdx.x; i < npieces; i += blockDim.x) {
        uintptr_t p = b16 + i * piece;
        size_t len = (e16 - p) < piece ? (e16 - p) : piece;
        prefetch_l2(reinterpret_cast<const void *>(p), static_cast<uint32_t>(len));
    }
}

__device__ __forceinline__ float silu_f32(float v)
{
    return v / (1.0f + expf(-v));
}

}  // namespace smoe
