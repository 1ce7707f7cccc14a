// Decode-time group-quantized GEMV kernels (one token): the fused gate/up
// pass and the down projection of a routed expert, Q4 and Q2.
//
// What they compute is fixed by the S-MoE page "Metal Compute Kernels",
// section "Fused FFN Kernels -- One Simdgroup Per Output Row":
//     hidden[i] = SiLU(gate . x)[i] * (up . x)[i]      (NMAT = 2)
//     out[j]    = (down . hidden)[j]                    (NMAT = 1)
// with w = (code - Z)(1/Z)s folded into an affine epilogue (qformat.cuh).
//
// This file holds the kernel for shapes the bulk-copy decode kernels
// (qgemv_reg.cu, qgemv_tma.cu) do not take: one warp per output row, its
// lanes striding over the row's 16-byte chunks, x staged once per CTA in
// swizzled shared memory, f32 arithmetic on the exact centred weights.
#include "common.cuh"
#include "internal.h"
#include "qformat.cuh"

namespace smoe {

struct QArgs {
    const uint8_t *codes[2];
    const float *scales[2];
    const float *x;
    float *y;
    int units;     // output rows
    int K;         // input length (columns)
    int group;     // columns per scale
};

// Any legal K: one warp per output row, lanes stride over the row's chunks.
template <int BITS, int NMAT>
__global__ void __launch_bounds__(256) qgemv_generic(QArgs a)
{
    using F = QFmt<BITS>;
    constexpr int F4W = F::CODES_PER_WORD / 4;
    extern __shared__ __align__(16) float4 smem4[];
    const int KC = a.K / F::CODES_PER_CHUNK;
    float4 *xs = smem4;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int ngroups = a.group > 0 ? a.K / a.group : 0;
    const int cpg = a.group / F::CODES_PER_CHUNK;
    const size_t row_bytes = static_cast<size_t>(KC) * 16;

    pdl_wait();
    stage_x_chunks<BITS>(a.x, a.K, xs);
    __syncthreads();
    pdl_launch_dependents();

    const uint32_t xs_base = smem_addr(xs);
    uint32_t xo[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) xo[m] = static_cast<uint32_t>(m ^ (lane & 7)) * 16u;

    for (int unit = blockIdx.x * nwarps + warp; unit < a.units; unit += gridDim.x * nwarps) {
        float acc[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) acc[m] = 0.f;
        for (int cc = lane; cc < KC; cc += 32) {
            uint4 cw[NMAT];
            float sc[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                cw[m] = ldg_stream(a.codes[m] + unit * row_bytes + static_cast<size_t>(cc) * 16);
                sc[m] = ldg_f32(a.scales[m] + static_cast<size_t>(unit) * ngroups + cc / cpg);
            }
            const uint32_t cbase = xs_base + static_cast<uint32_t>(cc * F::F4_PER_CHUNK) * 16u;
            float P[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) P[m] = 0.f;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                float xv[F::CODES_PER_WORD];
#pragma unroll
                for (int q = 0; q < F4W; ++q) {
                    const int m = wi * F4W + q;
                    const float4 v = lds128(cbase + static_cast<uint32_t>((m & 8) * 16) + xo[m & 7]);
                    xv[4 * q + 0] = v.x;
                    xv[4 * q + 1] = v.y;
                    xv[4 * q + 2] = v.z;
                    xv[4 * q + 3] = v.w;
                }
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    const uint32_t w = word_of(cw[m], wi);
#pragma unroll
                    for (int i = 0; i < F::CODES_PER_WORD; ++i)
                        P[m] = fmaf(code_centred<BITS>(w, i), xv[i], P[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m) acc[m] = fmaf(sc[m], P[m], acc[m]);
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(FULL_MASK, acc[m], off);
        if (lane == 0) {
            const float y0 = F::A * acc[0];
            if (NMAT == 2) {
                const float y1 = F::A * acc[NMAT - 1];
                a.y[unit] = silu_f32(y0) * y1;
            } else {
                a.y[unit] = y0;
            }
        }
    }
}

// ---------------------------------------------------------------- host side

namespace {

template <int BITS, int NMAT>
using QKernel = void (*)(QArgs);

template <int BITS, int NMAT>
cudaError_t launch_q(const QArgs &base, cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    QArgs a = base;
    const size_t smem = static_cast<size_t>(a.K) * sizeof(float);
    QKernel<BITS, NMAT> k = qgemv_generic<BITS, NMAT>;
    const int warps = 8;
    long long blocks = (static_cast<long long>(a.units) + warps - 1) / warps;
    const long long cap = static_cast<long long>(dev->sm_count) * 4;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(warps * 32), smem, stream, a);
}

}  // namespace

cudaError_t launch_qgemv(int bits, int nmat, const uint8_t *const codes[2],
                         const float *const scales[2], const float *x, float *y, int units,
                         int K, int group, cudaStream_t stream)
{
    QArgs a = {};
    a.codes[0] = codes[0];
    a.codes[1] = nmat == 2 ? codes[1] : codes[0];
    a.scales[0] = scales[0];
    a.scales[1] = nmat == 2 ? scales[1] : scales[0];
    a.x = x;
    a.y = y;
    a.units = units;
    a.K = K;
    a.group = group;
    // The bulk-copy kernel (qgemv_tma.cu) takes every shape whose rows are a
    // multiple of 8 chunks and whose staging fits in shared memory; the
    // kernels above serve the rest (narrow or ragged rows, K = 0).
    bool unsupported = true;
    const uint8_t *c1 = a.codes[1];
    const float *s1 = a.scales[1];
    cudaError_t e = launch_qgemv_experts(bits, nmat, 1, &a.codes[0], &c1, &a.scales[0], &s1, &a.x, &a.y, units,
                                         K, group, stream, &unsupported);
    if (!unsupported) return e;
    if (bits == 4) return nmat == 2 ? launch_q<4, 2>(a, stream) : launch_q<4, 1>(a, stream);
    return nmat == 2 ? launch_q<2, 2>(a, stream) : launch_q<2, 1>(a, stream);
}

}  // namespace smoe
