// The row-block sweep of the dense bf16 matvec (bf16_gemv.cu), shared by
// the matvec kernels and the fused router (route.cu).  The S-MoE page
// "Metal Compute Kernels", section "Coalesced Dense Matvec -- the Same
// Contract for bf16": y = W x with bf16 W, f32 x and y.
#pragma once

#include "common.cuh"

namespace smoe {

constexpr int BF_THREADS = 512;
constexpr int BF_WARPS = BF_THREADS / 32;
constexpr int BF_GMAX = 8;

// Rows [r0, r1) of y = W x by the whole CTA.  CPL: 16-byte chunks per
// thread per row (K <= CPL * 512 * 8).  xs: K floats of dynamic shared
// memory; part: the per-warp row sums.
template <int CPL>
__device__ __forceinline__ void bf16_rows(const uint16_t *__restrict__ w, const float *__restrict__ x,
                                          float *__restrict__ y, int r0, int r1, int K, uint32_t prefetch_bytes,
                                          float4 *xs, float (&part)[2][BF_WARPS][BF_GMAX])
{
    constexpr int BF_G = 8 / CPL > 2 ? 8 / CPL : 2;  // rows per group
    constexpr bool XREG = CPL <= 2;                 // x of the thread's chunks in registers
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int KC = K >> 3;  // 16-byte chunks per row
    const size_t row_elems = static_cast<size_t>(K);

    if (prefetch_bytes && r1 > r0) {
        size_t range = static_cast<size_t>(r1 - r0) * row_elems * 2;
        if (range > prefetch_bytes) range = prefetch_bytes;
        prefetch_range_l2(w + static_cast<size_t>(r0) * row_elems, range, 16384);
    }

    pdl_wait();
    const int nq = K >> 2;
    for (int q = t; q < nq; q += BF_THREADS) xs[q] = reinterpret_cast<const float4 *>(x)[q];
    __syncthreads();
    pdl_launch_dependents();

    // this thread's x for its chunks (zero past the row)
    auto x_of = [&](int j, float (&v)[8]) {
        const int cc = t + BF_THREADS * j;
        if (cc < KC) {
            const float4 x0 = xs[2 * cc], x1 = xs[2 * cc + 1];
            v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
            v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = 0.f;
        }
    };
    float xv[XREG ? CPL : 1][8];
#pragma unroll
    for (int j = 0; j < (XREG ? CPL : 1); ++j) x_of(j, xv[j]);

    // loads of one group: rows r .. r + G - 1 (rows past r1 read row r1 - 1)
    auto load_group = [&](int r, uint4 (&c)[BF_G][CPL]) {
#pragma unroll
        for (int g = 0; g < BF_G; ++g) {
            const int row = min(r + g, r1 - 1);
            const uint16_t *wrow = w + static_cast<size_t>(row) * row_elems;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int cc = t + BF_THREADS * j;
                c[g][j] = cc < KC ? ldg_stream(wrow + static_cast<size_t>(cc) * 8) : make_uint4(0, 0, 0, 0);
            }
        }
    };

    uint4 cur[BF_G][CPL], nxt[BF_G][CPL];
    if (r0 < r1) load_group(r0, cur);
    int buf = 0;
    for (int r = r0; r < r1; r += BF_G) {
        if (r + BF_G < r1) load_group(r + BF_G, nxt);
        float s[BF_G];
#pragma unroll
        for (int g = 0; g < BF_G; ++g) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const uint4 c = cur[g][j];
                float xl[8];
                if (XREG) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) xl[k] = xv[XREG ? j : 0][k];
                } else {
                    x_of(j, xl);
                }
                a0 = fmaf(__uint_as_float(c.x << 16), xl[0], a0);
                a1 = fmaf(__uint_as_float(c.x & 0xffff0000u), xl[1], a1);
                a0 = fmaf(__uint_as_float(c.y << 16), xl[2], a0);
                a1 = fmaf(__uint_as_float(c.y & 0xffff0000u), xl[3], a1);
                a0 = fmaf(__uint_as_float(c.z << 16), xl[4], a0);
                a1 = fmaf(__uint_as_float(c.z & 0xffff0000u), xl[5], a1);
                a0 = fmaf(__uint_as_float(c.w << 16), xl[6], a0);
                a1 = fmaf(__uint_as_float(c.w & 0xffff0000u), xl[7], a1);
            }
            s[g] = a0 + a1;
        }
        // warp sums of the G rows (butterfly: every lane ends with each sum);
        // lane g keeps row g's, then one thread per row adds the 16 warps'
#pragma unroll
        for (int g = 0; g < BF_G; ++g)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s[g] += __shfl_xor_sync(FULL_MASK, s[g], off);
        if (lane < BF_G) {
            float v = s[0];
#pragma unroll
            for (int g = 1; g < BF_G; ++g)
                if (lane == g) v = s[g];
            part[buf][warp][lane] = v;
        }
        __syncthreads();
        if (t < BF_G && r + t < r1) {
            float v = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < BF_WARPS; ++w2) v += part[buf][w2][t];
            y[r + t] = v;
        }
        buf ^= 1;
#pragma unroll
        for (int g = 0; g < BF_G; ++g)
#pragma unroll
            for (int j = 0; j < CPL; ++j) cur[g][j] = nxt[g][j];
    }
}

}  // namespace smoe
