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

namespace smoe {

// ---- mbarrier and bulk-copy (TMA engine) helpers, CTA-local shared memory.

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One bulk copy global -> shared, completing `bytes` of transaction count on
// the mbarrier.  dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Tests phase `parity` of an mbarrier.  While the phase is incomplete the
// hardware may suspend the thread for up to about 20 us (the suspend-time
// hint) and wakes it when the phase completes, so waiting warps leave the
// issue slots and the shared-memory pipe to the warps that have work.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, 20000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Arrives once on an mbarrier (release, CTA scope).
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32) of the block.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Waits for phase `parity` of an mbarrier, giving up after about two seconds
// of SM clock (or 2^24 polls); on giving up it records `code` in *status
// (if not null) and returns false instead of hanging.  Between polls the
// thread sleeps briefly so that waiting warps leave the issue slots to the
// warps that have work.  A parity test cannot tell a phase from the one two
// before it, so the caller must know that the phase preceding the awaited
// one has already completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned *status,
                                                  unsigned code)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        __nanosleep(64);
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > 4000000000LL) break;
    }
    if (status) atomicExch(status, code);
    return false;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits (bounded, about two seconds of SM clock) until *p >= target.
__device__ __forceinline__ bool wait_count(const unsigned *p, unsigned target)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const long long t0 = clock64();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        __nanosleep(128);
        if (ld_acquire_gpu(p) >= target) return true;
        if (clock64() - t0 > 4000000000LL) break;
    }
    return false;
}

}  // namespace smoe
