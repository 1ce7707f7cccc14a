// Decode-time group-quantized GEMV kernels (one token): the fused gate/up
// pass and the down projection of a routed expert, Q4 and Q2.
//
// What they compute is fixed by the S-MoE page "Metal Compute Kernels",
// section "Fused FFN Kernels -- One Simdgroup Per Output Row":
//     hidden[i] = SiLU(gate . x)[i] * (up . x)[i]      (NMAT = 2)
//     out[j]    = (down . hidden)[j]                    (NMAT = 1)
// with w = (code - Z)(1/Z)s folded into an affine epilogue (qformat.cuh).
//
// GB300 layout (not the page's Metal layout):
//  * a "team" of L lanes (L = 8, 16 or 32) owns one output row at a time and
//    reads it as 16-byte chunks; consecutive teams own consecutive rows, so a
//    warp's load instruction covers whole 128-byte lines;
//  * each team holds RPT rows (and, for gate/up, the gate and the up row of
//    the same output) at once, so every x value read from shared memory
//    feeds NMAT * RPT FMAs;
//  * all code chunks of a row tile are loaded before any is used (up to
//    NMAT * RPT * CPL 16-byte loads in flight per lane);
//  * one CTA per SM owns a contiguous, balanced range of row tiles; before
//    waiting on the previous kernel it issues bulk L2 prefetches of its
//    whole weight range, so HBM traffic starts while x is still unknown;
//  * x is staged once per CTA in swizzled shared memory.
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
    int tiles;     // row tiles (fast kernel)
    int prefetch;  // issue the bulk L2 prefetch of this CTA's weights
};

constexpr uint32_t PREFETCH_PIECE = 16384;

// Fast path: every row is exactly L * CPL chunks (K == L*CPL*CODES_PER_CHUNK).
template <int BITS, int L, int CPL, int RPT, int NMAT>
__global__ void __launch_bounds__(256) qgemv_fast(QArgs a)
{
    using F = QFmt<BITS>;
    constexpr int TEAMS = 32 / L;
    constexpr int UPT = TEAMS * RPT;  // output rows per warp tile
    constexpr int KC = L * CPL;       // chunks per row
    constexpr int ROW_BYTES = KC * 16;
    constexpr int F4W = F::CODES_PER_WORD / 4;  // float4s of x per code word
    static_assert(L == 8 || L == 16 || L == 32, "team size");

    extern __shared__ __align__(16) float4 smem4[];
    float4 *xs = smem4;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int team = lane / L;
    const int u = lane % L;
    const int ngroups = a.K / a.group;
    const int cpg = a.group / F::CODES_PER_CHUNK;  // chunks per group

    const int t0 = static_cast<int>(static_cast<long long>(a.tiles) * blockIdx.x / gridDim.x);
    const int t1 = static_cast<int>(static_cast<long long>(a.tiles) * (blockIdx.x + 1) / gridDim.x);

    if (a.prefetch) {
        const int u0 = t0 * UPT;
        const int u1 = min(a.units, t1 * UPT);
        if (u1 > u0) {
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                prefetch_range_l2(a.codes[m] + static_cast<size_t>(u0) * ROW_BYTES,
                                  static_cast<size_t>(u1 - u0) * ROW_BYTES, PREFETCH_PIECE);
                prefetch_range_l2(a.scales[m] + static_cast<size_t>(u0) * ngroups,
                                  static_cast<size_t>(u1 - u0) * ngroups * sizeof(float),
                                  PREFETCH_PIECE);
            }
        }
    }

    pdl_wait();
    stage_x_chunks<BITS>(a.x, a.K, xs);
    __syncthreads();
    pdl_launch_dependents();

    // Shared-memory addresses of the 8 swizzled float4 slots this lane reads
    // inside each of its chunks (chunk index = u + L*j, so chunk & 7 = u & 7).
    const uint32_t xs_base = smem_addr(xs);
    uint32_t xb[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
        xb[m] = xs_base + static_cast<uint32_t>(u * F::F4_PER_CHUNK + (m ^ (u & 7))) * 16u;
    int gidx[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) gidx[j] = (u + L * j) / cpg;

    for (int tile = t0 + warp; tile < t1; tile += nwarps) {
        uint4 cw[NMAT][RPT][CPL];
        float sc[NMAT][RPT][CPL];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int unit = tile * UPT + r * TEAMS + team;
            const bool ok = unit < a.units;
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const uint8_t *row = a.codes[m] + static_cast<size_t>(unit) * ROW_BYTES + u * 16;
                const float *srow = a.scales[m] + static_cast<size_t>(unit) * ngroups;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    cw[m][r][j] = ok ? ldg_stream(row + L * 16 * j) : make_uint4(0, 0, 0, 0);
                    sc[m][r][j] = ok ? ldg_f32(srow + gidx[j]) : 0.f;
                }
            }
        }

        float acc[NMAT][RPT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r) acc[m][r] = 0.f;

#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            float P[NMAT][RPT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int r = 0; r < RPT; ++r) P[m][r] = 0.f;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                float xv[F::CODES_PER_WORD];
#pragma unroll
                for (int q = 0; q < F4W; ++q) {
                    const int m = wi * F4W + q;  // float4 index inside the chunk
                    const float4 v = lds128(xb[m & 7] + static_cast<uint32_t>(((m & 8) + L * j * F::F4_PER_CHUNK) * 16));
                    xv[4 * q + 0] = v.x;
                    xv[4 * q + 1] = v.y;
                    xv[4 * q + 2] = v.z;
                    xv[4 * q + 3] = v.w;
                }
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int r = 0; r < RPT; ++r) {
                        const uint32_t w = word_of(cw[m][r][j], wi);
#pragma unroll
                        for (int i = 0; i < F::CODES_PER_WORD; ++i)
                            P[m][r] = fmaf(code_centred<BITS>(w, i), xv[i], P[m][r]);
                    }
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    acc[m][r] = fmaf(sc[m][r][j], P[m][r], acc[m][r]);
                }
        }

#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
                for (int off = L / 2; off > 0; off >>= 1) acc[m][r] += __shfl_xor_sync(FULL_MASK, acc[m][r], off);

        if (u == 0) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int unit = tile * UPT + r * TEAMS + team;
                if (unit < a.units) {
                    const float y0 = F::A * acc[0][r];
                    if (NMAT == 2) {
                        const float y1 = F::A * acc[NMAT - 1][r];
                        a.y[unit] = silu_f32(y0) * y1;
                    } else {
                        a.y[unit] = y0;
                    }
                }
            }
        }
    }
}

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

struct FastPick {
    int L, CPL;
};

// (L, CPL) pairs the fast kernel is built for; the first whose L*CPL equals
// the chunk count of a row is used.
constexpr FastPick kFastPicks[] = {{32, 4}, {32, 3}, {32, 2}, {32, 1}, {16, 3},
                                   {16, 1}, {8, 3},  {8, 1}};

template <int BITS, int NMAT>
QKernel<BITS, NMAT> fast_kernel(int L, int CPL)
{
    constexpr int RPT = 1;
    // Q2 chunks carry 64 codes; more than two per lane exhaust the registers.
    constexpr int MAXCPL = BITS == 4 ? 4 : 2;
    if (L == 32 && CPL == 4) return MAXCPL >= 4 ? qgemv_fast<BITS, 32, (MAXCPL >= 4 ? 4 : 1), RPT, NMAT> : nullptr;
    if (L == 32 && CPL == 3) return MAXCPL >= 3 ? qgemv_fast<BITS, 32, (MAXCPL >= 3 ? 3 : 1), RPT, NMAT> : nullptr;
    if (L == 32 && CPL == 2) return qgemv_fast<BITS, 32, 2, RPT, NMAT>;
    if (L == 32 && CPL == 1) return qgemv_fast<BITS, 32, 1, RPT, NMAT>;
    if (L == 16 && CPL == 3) return MAXCPL >= 3 ? qgemv_fast<BITS, 16, (MAXCPL >= 3 ? 3 : 1), RPT, NMAT> : nullptr;
    if (L == 16 && CPL == 1) return qgemv_fast<BITS, 16, 1, RPT, NMAT>;
    if (L == 8 && CPL == 3) return MAXCPL >= 3 ? qgemv_fast<BITS, 8, (MAXCPL >= 3 ? 3 : 1), RPT, NMAT> : nullptr;
    if (L == 8 && CPL == 1) return qgemv_fast<BITS, 8, 1, RPT, NMAT>;
    return nullptr;
}

template <int BITS, int NMAT>
cudaError_t launch_q(const QArgs &base, cudaStream_t stream)
{
    using F = QFmt<BITS>;
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    QArgs a = base;
    const int KC = a.K / F::CODES_PER_CHUNK;
    const size_t smem = static_cast<size_t>(a.K) * sizeof(float);
    constexpr int RPT = 1;

    for (const FastPick &p : kFastPicks) {
        if (p.L * p.CPL != KC) continue;
        QKernel<BITS, NMAT> k = fast_kernel<BITS, NMAT>(p.L, p.CPL);
        if (!k) break;
        const int upt = (32 / p.L) * RPT;
        a.tiles = (a.units + upt - 1) / upt;
        int grid = a.tiles < dev->sm_count ? a.tiles : dev->sm_count;
        const int per_cta = (a.tiles + grid - 1) / grid;
        int warps = per_cta < 4 ? 4 : (per_cta > 8 ? 8 : per_cta);
        a.prefetch = 1;
        cudaError_t e = ensure_dynamic_smem(k, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(k, dim3(grid), dim3(warps * 32), smem, stream, a);
    }

    QKernel<BITS, NMAT> k = qgemv_generic<BITS, NMAT>;
    const int warps = 8;
    long long blocks = (static_cast<long long>(a.units) + warps - 1) / warps;
    const long long cap = static_cast<long long>(dev->sm_count) * 4;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    a.tiles = 0;
    a.prefetch = 0;
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
