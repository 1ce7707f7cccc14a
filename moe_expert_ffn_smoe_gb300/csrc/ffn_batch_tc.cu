// Token-batch FFN on the tensor cores (tcgen05, TMEM), the S-MoE page "Metal
// Compute Kernels", section "Token-Batch Fused FFN": for T tokens the three
// projections are dense contractions, Y = W X^T with the weights' K axis
// contracted against every token.
//
// Exactness plan (the scale varies per (row, group), so it cannot be folded
// into an operand):
//  * A (weights, M x 64 per group slice) holds each code c as the bf16 value
//    1 + c/16, which is exact.  The affine fold then reads, per 64-column
//    tile of one group, D = sum (1 + c/16) x = Sx + C/16 and
//        sum w x = s (C/Z - Sx) = s (A D - (A + 1) Sx),   A = 16/Z.
//  * B (tokens, N x 64) holds x split into two bf16 halves, hi = bf16(x) and
//    lo = bf16(x - hi); two MMAs accumulate D over hi and lo into the same
//    TMEM accumulator (x represented to about 2^-17 relative), and Sx is the
//    f32 sum of hi + lo over the tile, so D and Sx see the same x.
//  * Each 64-column tile's accumulator is read back from TMEM and folded
//    into per-thread f32 sums with the tile's scale (double-buffered, so the
//    next tile's MMAs run while the epilogue reads this one).
//
// CTA roles (288 threads): warps 0-3 epilogue (TMEM lane quarters 0-3 =
// rows 0-127), warps 4-7 operand preparation (unpack codes to bf16 in the
// canonical no-swizzle K-major layout, bulk-copy the pre-split token block),
// warp 8 MMA issue and TMEM allocation.  Stages of shared memory hand tiles
// from the preparation warps to the MMA thread ("full" barriers) and back
// ("empty", signalled by tcgen05.commit); two TMEM buffers hand accumulators
// to the epilogue and back.  Every barrier has one in-order waiter, so the
// parity of each awaited phase is unambiguous; every wait is bounded.
//
// Grid: (matrix x 128-row tile, token tile, K split).  With a K split the
// partial sums are added into a zero-initialised output with f32 atomics.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace smoe {
namespace {

constexpr int KT = 64;   // columns per K tile (one group slice)
constexpr int MT = 128;  // rows per CTA tile
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 4;
constexpr int PREP_WARPS = 4;
constexpr int TC_THREADS = (EPI_WARPS + PREP_WARPS + 1) * 32;
constexpr uint32_t A_BYTES = MT * KT * 2;
constexpr float FOLD_A = 16.0f / 7.5f;

__host__ __device__ constexpr uint32_t b_bytes(int nt) { return static_cast<uint32_t>(nt) * KT * 2u * 2u; }
__host__ __device__ constexpr uint32_t stage_bytes(int nt) { return A_BYTES + b_bytes(nt); }

// Byte offset of (row, 8-column block k8) in a [rows x 64] bf16 tile laid out
// as 8x8 core matrices: core (row/8, k8) at ((row/8)*8 + k8)*128, row%8 at 16*(row%8).
__device__ __forceinline__ uint32_t core_off(int row, int k8)
{
    return static_cast<uint32_t>(((row >> 3) * 8 + k8) * 128 + (row & 7) * 16);
}

// Inside every 8-column block the K order is 0,4,1,5,2,6,3,7 (the order in
// which a 32-bit word of Q4 codes unpacks to bf16 pairs); B uses the same
// order, so the contraction is unchanged.
__device__ __forceinline__ int perm8(int p) { return (p & 1) ? 4 + (p >> 1) : (p >> 1); }

// tcgen05 shared-memory matrix descriptor, no swizzle, K-major:
// LBO = distance between core matrices along K (128 B), SBO = between 8-row
// groups (1024 B), version field 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
           (static_cast<uint64_t>(1024u >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor, kind::f16: f32 accumulate, A and B bf16, both
// K-major, N at bit 17 (in 8s), M at bit 24 (in 16s).
__host__ __device__ constexpr uint32_t instr_desc(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive f32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// One 32-bit word of Q4 codes (columns 0..7) as 8 exact bf16 values
// 1 + c/16, in the order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ uint4 q4_word_to_bf16(uint32_t w)
{
    const uint32_t mag = 0x3F803F80u;
    uint4 r;
    r.x = ((w << 3) & 0x00780078u) | mag;  // columns 0 and 4
    r.y = ((w >> 1) & 0x00780078u) | mag;  // 1 and 5
    r.z = ((w >> 5) & 0x00780078u) | mag;  // 2 and 6
    r.w = ((w >> 9) & 0x00780078u) | mag;  // 3 and 7
    return r;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- B prep

struct PrepArgs {
    const float *X;  // mode 0: [T x K]
    const float *G;  // mode 1: [T x K] pre-activation gate sums
    const float *U;  //         [T x K] up sums
    uint8_t *Bblk;   // [T/nt][K/64] blocks of b_bytes(nt): hi then lo
    float *Sx;       // [K/64][Tpad]
    int T, Tpad, K, nt, mode;
};

// One thread per (token, 8-column block): the token's 8 values (or SiLU(g)*u)
// split into bf16 hi/lo in the tile layout, plus the per-tile sums of hi+lo.
__global__ void __launch_bounds__(256) prep_b(PrepArgs a)
{
    pdl_wait();
    const int kb_per_t = a.K / 8;
    const int nkt = a.K / KT;
    const long long total = static_cast<long long>(a.Tpad) * kb_per_t;  // multiple of 8
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long rounds = (total + stride - 1) / stride;
    for (long long rd = 0; rd < rounds; ++rd) {
        const long long idx = rd * stride + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
        float part = 0.f;
        int t = 0, kt = 0;
        const bool live = idx < total;
        if (live) {
            t = static_cast<int>(idx / kb_per_t);
            const int kb = static_cast<int>(idx % kb_per_t);
            kt = kb / 8;
            const int k8 = kb % 8;
            float v[8];
            if (t < a.T) {
                const size_t base = static_cast<size_t>(t) * a.K + static_cast<size_t>(kb) * 8;
                float raw[8];
                if (a.mode == 0) {
                    const float4 p0 = reinterpret_cast<const float4 *>(a.X + base)[0];
                    const float4 p1 = reinterpret_cast<const float4 *>(a.X + base)[1];
                    raw[0] = p0.x; raw[1] = p0.y; raw[2] = p0.z; raw[3] = p0.w;
                    raw[4] = p1.x; raw[5] = p1.y; raw[6] = p1.z; raw[7] = p1.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) raw[i] = silu_f32(a.G[base + i]) * a.U[base + i];
                }
#pragma unroll
                for (int p = 0; p < 8; ++p) v[p] = raw[perm8(p)];
            } else {
#pragma unroll
                for (int p = 0; p < 8; ++p) v[p] = 0.f;
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int p = 0; p < 8; p += 2) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(v[p]);
                const __nv_bfloat16 h1 = __float2bfloat16_rn(v[p + 1]);
                const float r0 = v[p] - __bfloat162float(h0);
                const float r1 = v[p + 1] - __bfloat162float(h1);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(r0);
                const __nv_bfloat16 l1 = __float2bfloat16_rn(r1);
                part += (__bfloat162float(h0) + __bfloat162float(l0)) + (__bfloat162float(h1) + __bfloat162float(l1));
                hi[p / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
                lo[p / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
            }
            uint8_t *blk = a.Bblk + (static_cast<size_t>(t / a.nt) * nkt + kt) * b_bytes(a.nt);
            const uint32_t off = core_off(t % a.nt, k8);
            *reinterpret_cast<uint4 *>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(blk + static_cast<size_t>(a.nt) * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // the 8 blocks of one (token, K tile) are 8 consecutive threads
        part += __shfl_xor_sync(FULL_MASK, part, 1);
        part += __shfl_xor_sync(FULL_MASK, part, 2);
        part += __shfl_xor_sync(FULL_MASK, part, 4);
        if (live && (idx % 8) == 0) a.Sx[static_cast<size_t>(kt) * a.Tpad + t] = part;
    }
    pdl_launch_dependents();
}

// ---------------------------------------------------------------- GEMM

struct TcArgs {
    const uint8_t *codes[2];
    const float *scales[2];
    float *out[2];  // [T x M] per matrix
    const uint8_t *Bblk;
    const float *Sx;
    unsigned *status;
    int M, K, group, T, Tpad;
    int mtiles;        // 128-row tiles per matrix
    int kt_per_split;  // K tiles per CTA
    int atomic;        // K split: accumulate into zeroed outputs
};

template <int NT>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm(const __grid_constant__ TcArgs a)
{
    constexpr uint32_t NCOLS = (2 * NT) < 32 ? 32 : 2 * NT;  // two accumulator buffers
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + STAGES * stage_bytes(NT);
    const uint32_t full0 = bars, empty0 = bars + 8 * STAGES, accf0 = bars + 16 * STAGES,
                   acce0 = accf0 + 16, tslot = acce0 + 16;
    uint32_t *tmem_word = reinterpret_cast<uint32_t *>(smem_raw + (tslot - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x / a.mtiles;
    const int row0 = (blockIdx.x % a.mtiles) * MT;
    const int ntile = blockIdx.y;
    const int nkt = a.K / KT;
    const int kt0 = blockIdx.z * a.kt_per_split;
    const int kt1 = min(nkt, kt0 + a.kt_per_split);
    const int nk = kt1 > kt0 ? kt1 - kt0 : 0;
    const int ngroups = a.K / a.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, PREP_WARPS + 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, EPI_WARPS);
        }
        fence_mbar_init();
    }
    if (warp == EPI_WARPS + PREP_WARPS) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(NCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_word;
    pdl_wait();

    if (warp == EPI_WARPS + PREP_WARPS) {
        // ---- MMA issue
        if (lane == 0) {
            const uint32_t idesc = instr_desc(MT, NT);
            for (int i = 0; i < nk; ++i) {
                const int s = i % STAGES;
                const int b = i & 1;
                if (!mbar_wait_bounded(full0 + 8 * s, (i / STAGES) & 1, a.status, 3u)) break;
                if (i >= 2 && !mbar_wait_bounded(acce0 + 8 * b, ((i >> 1) - 1) & 1, a.status, 4u)) break;
                tc_fence_after();
                const uint32_t sa = base + s * stage_bytes(NT);
                const uint32_t sb = sa + A_BYTES;
                const uint32_t d = tmem + static_cast<uint32_t>(b * NT);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk)
                        mma_bf16(d, smem_desc(sa + kk * 256), smem_desc(sb + part * NT * 128 + kk * 256), idesc,
                                 (part | kk) != 0);
                mma_commit(empty0 + 8 * s);
                mma_commit(accf0 + 8 * b);
            }
        }
    } else if (warp >= EPI_WARPS) {
        // ---- operand preparation: thread pi owns row pi of the tile
        const int pi = threadIdx.x - EPI_WARPS * 32;
        const int row = row0 + pi;
        const bool rok = row < a.M;
        const size_t row_bytes = static_cast<size_t>(a.K) / 2;
        const uint8_t *crow = a.codes[m] + static_cast<size_t>(rok ? row : 0) * row_bytes;
        const uint8_t *bsrc = a.Bblk + static_cast<size_t>(ntile) * nkt * b_bytes(NT);
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
        if (nk > 0 && rok) {
            c0 = ldg_u4(crow + static_cast<size_t>(kt0) * 32);
            c1 = ldg_u4(crow + static_cast<size_t>(kt0) * 32 + 16);
        }
        for (int i = 0; i < nk; ++i) {
            const int s = i % STAGES;
            if (i >= STAGES && !mbar_wait_bounded(empty0 + 8 * s, ((i / STAGES) - 1) & 1, a.status, 5u)) break;
            const uint32_t sa = base + s * stage_bytes(NT);
            if (pi == 0) {
                mbar_arrive_expect_tx(full0 + 8 * s, b_bytes(NT));
                bulk_g2s(sa + A_BYTES, bsrc + static_cast<size_t>(kt0 + i) * b_bytes(NT), b_bytes(NT), full0 + 8 * s);
            }
            const uint4 w0 = c0, w1 = c1;
            if (i + 1 < nk && rok) {  // next tile's codes while this one is unpacked
                c0 = ldg_u4(crow + static_cast<size_t>(kt0 + i + 1) * 32);
                c1 = ldg_u4(crow + static_cast<size_t>(kt0 + i + 1) * 32 + 16);
            }
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) sts128(sa + core_off(pi, k8), q4_word_to_bf16(rok ? words[k8] : 0u));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * s);
        }
    } else {
        // ---- epilogue: warp q reads TMEM lanes 32q..32q+31 (= tile rows)
        const int r = warp * 32 + lane;
        const int row = row0 + r;
        const bool rok = row < a.M;
        float y[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) y[n] = 0.f;
        const float *srow = a.scales[m] + static_cast<size_t>(rok ? row : 0) * ngroups;
        for (int i = 0; i < nk; ++i) {
            const int b = i & 1;
            const int kt = kt0 + i;
            const float sc = rok ? ldg_f32(srow + (kt * KT) / a.group) : 0.f;
            const bool ok = mbar_wait_bounded(accf0 + 8 * b, (i >> 1) & 1, a.status, 6u);
            if (!__all_sync(FULL_MASK, ok)) break;
            tc_fence_after();
            float d[NT];
#pragma unroll
            for (int c = 0; c < NT; c += 16) {
                float v[16];
                tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(b * NT + c), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) d[c + j] = v[j];
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * b);
            const float *sx = a.Sx + static_cast<size_t>(kt) * a.Tpad + static_cast<size_t>(ntile) * NT;
            const float sa = sc * FOLD_A, sb = sc * (FOLD_A + 1.0f);
#pragma unroll
            for (int n = 0; n < NT; n += 4) {
                const float4 s4 = *reinterpret_cast<const float4 *>(sx + n);
                y[n + 0] = fmaf(sa, d[n + 0], fmaf(-sb, s4.x, y[n + 0]));
                y[n + 1] = fmaf(sa, d[n + 1], fmaf(-sb, s4.y, y[n + 1]));
                y[n + 2] = fmaf(sa, d[n + 2], fmaf(-sb, s4.z, y[n + 2]));
                y[n + 3] = fmaf(sa, d[n + 3], fmaf(-sb, s4.w, y[n + 3]));
            }
        }
        if (rok && nk > 0) {
            float *o = a.out[m];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int t = ntile * NT + n;
                if (t < a.T) {
                    if (a.atomic) atomicAdd(o + static_cast<size_t>(t) * a.M + row, y[n]);
                    else o[static_cast<size_t>(t) * a.M + row] = y[n];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (warp == EPI_WARPS + PREP_WARPS) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOLS) : "memory");
    }
}

int pick_nt(int T) { return T > 32 ? 64 : (T > 16 ? 32 : 16); }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct TcLayout {
    int nt, Tpad;
    size_t xb, sx, g, u, hb, sh, total;
};

TcLayout tc_layout(int T, int d_model, int d_ff)
{
    TcLayout L = {};
    L.nt = pick_nt(T);
    L.Tpad = (T + L.nt - 1) / L.nt * L.nt;
    size_t off = 0;
    L.xb = off; off = align256(off + static_cast<size_t>(L.Tpad) * d_model * 4);
    L.sx = off; off = align256(off + static_cast<size_t>(d_model / KT) * L.Tpad * 4);
    L.g = off;  off = align256(off + static_cast<size_t>(T) * d_ff * 4);
    L.u = off;  off = align256(off + static_cast<size_t>(T) * d_ff * 4);
    L.hb = off; off = align256(off + static_cast<size_t>(L.Tpad) * d_ff * 4);
    L.sh = off; off = align256(off + static_cast<size_t>(d_ff / KT) * L.Tpad * 4);
    L.total = off;
    return L;
}

template <int NT>
cudaError_t launch_gemm(TcArgs a, int nmat, int ntiles, int sms, cudaStream_t stream)
{
    const int nkt = a.K / KT;
    const int base_ctas = nmat * a.mtiles * ntiles;
    int ks = sms / (base_ctas > 0 ? base_ctas : 1);
    if (ks < 1) ks = 1;
    if (ks > nkt) ks = nkt;
    a.kt_per_split = (nkt + ks - 1) / ks;
    ks = (nkt + a.kt_per_split - 1) / a.kt_per_split;
    a.atomic = ks > 1;
    if (a.atomic) {
        for (int i = 0; i < nmat; ++i) {
            cudaError_t e = cudaMemsetAsync(a.out[i], 0, static_cast<size_t>(a.T) * a.M * sizeof(float), stream);
            if (e != cudaSuccess) return e;
        }
    }
    const size_t smem = 1024 + STAGES * stage_bytes(NT) + 256;
    auto k = tc_gemm<NT>;
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(nmat * a.mtiles, ntiles, ks), dim3(TC_THREADS), smem, stream, a);
}

cudaError_t launch_gemm_nt(int nt, const TcArgs &a, int nmat, int ntiles, int sms, cudaStream_t stream)
{
    if (nt == 64) return launch_gemm<64>(a, nmat, ntiles, sms, stream);
    if (nt == 32) return launch_gemm<32>(a, nmat, ntiles, sms, stream);
    return launch_gemm<16>(a, nmat, ntiles, sms, stream);
}

cudaError_t launch_prep(PrepArgs p, int sms, cudaStream_t stream)
{
    const long long total = static_cast<long long>(p.Tpad) * (p.K / 8);
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(prep_b, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

}  // namespace

bool tc_batch_supported(int T, int d_model, int d_ff, int group)
{
    return T >= 2 && group % KT == 0 && d_model % KT == 0 && d_ff % KT == 0 && d_model > 0 && d_ff > 0;
}

size_t tc_batch_workspace(int T, int d_model, int d_ff)
{
    return tc_layout(T, d_model, d_ff).total;
}

cudaError_t launch_ffn_batch_tc(const uint8_t *const gu_codes[2], const float *const gu_scales[2],
                                const uint8_t *down_codes, const float *down_scales, const float *X, float *Y,
                                int T, int d_model, int d_ff, int group, void *workspace, cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const TcLayout L = tc_layout(T, d_model, d_ff);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *G = reinterpret_cast<float *>(ws + L.g);
    float *U = reinterpret_cast<float *>(ws + L.u);
    const int ntiles = L.Tpad / L.nt;

    PrepArgs p = {X, nullptr, nullptr, ws + L.xb, reinterpret_cast<float *>(ws + L.sx), T, L.Tpad, d_model, L.nt, 0};
    cudaError_t e = launch_prep(p, dev->sm_count, stream);
    if (e != cudaSuccess) return e;

    TcArgs a = {};
    a.codes[0] = gu_codes[0];
    a.codes[1] = gu_codes[1];
    a.scales[0] = gu_scales[0];
    a.scales[1] = gu_scales[1];
    a.out[0] = G;
    a.out[1] = U;
    a.Bblk = ws + L.xb;
    a.Sx = reinterpret_cast<const float *>(ws + L.sx);
    a.status = device_status_word();
    a.M = d_ff;
    a.K = d_model;
    a.group = group;
    a.T = T;
    a.Tpad = L.Tpad;
    a.mtiles = (d_ff + MT - 1) / MT;
    e = launch_gemm_nt(L.nt, a, 2, ntiles, dev->sm_count, stream);
    if (e != cudaSuccess) return e;

    PrepArgs q = {nullptr, G, U, ws + L.hb, reinterpret_cast<float *>(ws + L.sh), T, L.Tpad, d_ff, L.nt, 1};
    e = launch_prep(q, dev->sm_count, stream);
    if (e != cudaSuccess) return e;

    TcArgs b = a;
    b.codes[0] = b.codes[1] = down_codes;
    b.scales[0] = b.scales[1] = down_scales;
    b.out[0] = b.out[1] = Y;
    b.Bblk = ws + L.hb;
    b.Sx = reinterpret_cast<const float *>(ws + L.sh);
    b.M = d_model;
    b.K = d_ff;
    b.mtiles = (d_model + MT - 1) / MT;
    return launch_gemm_nt(L.nt, b, 1, ntiles, dev->sm_count, stream);
}

}  // namespace smoe
