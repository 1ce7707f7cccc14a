// Dense bf16 matvec y = W x (f32 x and y), the S-MoE page "Metal Compute
// Kernels", section "Coalesced Dense Matvec -- the Same Contract for bf16".
//
// GB300 layout: one warp per output row at a time; each lane reads 16-byte
// chunks (8 bf16) of the row, SEG chunks per lane per step, all issued before
// any is used.  A CTA owns a contiguous range of rows and bulk-prefetches the
// head of that range into L2 before waiting on the previous kernel.  x is
// staged once per CTA in swizzled shared memory.  A bf16 is the upper half
// of an f32, so widening is a shift or a mask: no conversion instruction.
#include "common.cuh"
#include "internal.h"

namespace smoe {

struct Bf16Args {
    const uint16_t *w;
    const float *x;
    float *y;
    int rows;
    int K;
    uint32_t prefetch_bytes;  // per CTA, from the start of its row range
};

// float4 slot of logical float4 q of x (bijection inside aligned blocks of
// eight float4s; lanes reading chunk = base + lane land in distinct banks).
__device__ __forceinline__ int bx_slot(int q) { return q ^ ((q >> 3) & 7); }

template <int SEG>
__global__ void __launch_bounds__(512) bf16_gemv(Bf16Args a)
{
    extern __shared__ __align__(16) float4 xs[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int KC = a.K >> 3;  // 16-byte chunks per row
    const size_t row_elems = static_cast<size_t>(a.K);

    const int r0 = static_cast<int>(static_cast<long long>(a.rows) * blockIdx.x / gridDim.x);
    const int r1 = static_cast<int>(static_cast<long long>(a.rows) * (blockIdx.x + 1) / gridDim.x);

    if (a.prefetch_bytes && r1 > r0) {
        size_t range = static_cast<size_t>(r1 - r0) * row_elems * 2;
        if (range > a.prefetch_bytes) range = a.prefetch_bytes;
        prefetch_range_l2(a.w + static_cast<size_t>(r0) * row_elems, range, 16384);
    }

    pdl_wait();
    const int nq = a.K >> 2;
    for (int q = threadIdx.x; q < nq; q += blockDim.x)
        xs[bx_slot(q)] = reinterpret_cast<const float4 *>(a.x)[q];
    __syncthreads();
    pdl_launch_dependents();

    // chunk cc = base + lane (base a multiple of 32) covers float4s 2cc, 2cc+1;
    // their slots are 2*base + ((2*lane + h) ^ ((lane >> 2) & 7)).
    const uint32_t xs_base = smem_addr(xs);
    const uint32_t xo0 = xs_base + static_cast<uint32_t>(((2 * lane) ^ ((lane >> 2) & 7)) * 16);
    const uint32_t xo1 = xs_base + static_cast<uint32_t>(((2 * lane + 1) ^ ((lane >> 2) & 7)) * 16);

    for (int row = r0 + warp; row < r1; row += nwarps) {
        const uint16_t *wrow = a.w + static_cast<size_t>(row) * row_elems;
        float acc0 = 0.f, acc1 = 0.f;
        for (int base = 0; base < KC; base += 32 * SEG) {
            uint4 c[SEG];
#pragma unroll
            for (int j = 0; j < SEG; ++j) {
                const int cc = base + lane + 32 * j;
                c[j] = cc < KC ? ldg_stream(wrow + static_cast<size_t>(cc) * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < SEG; ++j) {
                const int cb = base + 32 * j;  // chunk index of lane 0
                if (cb + lane < KC) {
                    const uint32_t off = static_cast<uint32_t>(cb) * 32u;  // 2*cb float4s
                    const float4 x0 = lds128(xo0 + off);
                    const float4 x1 = lds128(xo1 + off);
                    acc0 = fmaf(__uint_as_float(c[j].x << 16), x0.x, acc0);
                    acc1 = fmaf(__uint_as_float(c[j].x & 0xffff0000u), x0.y, acc1);
                    acc0 = fmaf(__uint_as_float(c[j].y << 16), x0.z, acc0);
                    acc1 = fmaf(__uint_as_float(c[j].y & 0xffff0000u), x0.w, acc1);
                    acc0 = fmaf(__uint_as_float(c[j].z << 16), x1.x, acc0);
                    acc1 = fmaf(__uint_as_float(c[j].z & 0xffff0000u), x1.y, acc1);
                    acc0 = fmaf(__uint_as_float(c[j].w << 16), x1.z, acc0);
                    acc1 = fmaf(__uint_as_float(c[j].w & 0xffff0000u), x1.w, acc1);
                }
            }
        }
        float acc = acc0 + acc1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, off);
        if (lane == 0) a.y[row] = acc;
    }
}

cudaError_t launch_bf16_gemv(const uint16_t *w, const float *x, float *y, int rows, int K,
                             cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    constexpr int SEG = 8;
    Bf16Args a = {w, x, y, rows, K, 0};
    // Shared memory rounded up to whole blocks of eight float4s (the swizzle
    // permutes inside such blocks).
    const size_t smem = ((static_cast<size_t>(K) / 4 + 7) / 8) * 8 * sizeof(float4);
    const int warps = 16;
    long long grid = dev->sm_count;
    const long long by_rows = (static_cast<long long>(rows) + 3) / 4;  // >= 4 rows per CTA
    if (by_rows < grid) grid = by_rows < 1 ? 1 : by_rows;
    // Prefetch at most 1/4 of L2's worth across the grid.
    const size_t l2_share = static_cast<size_t>(32u << 20) / static_cast<size_t>(grid);
    a.prefetch_bytes = static_cast<uint32_t>(l2_share < (1u << 20) ? l2_share : (1u << 20));
    auto k = bf16_gemv<SEG>;
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(static_cast<unsigned>(grid)), dim3(warps * 32), smem, stream, a);
}

}  // namespace smoe
