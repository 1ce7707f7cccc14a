// Shared pieces of the two decode kernels (qgemv_tma.cu: x digits read from
// shared memory; qgemv_reg.cu: x digits held in registers): the launch
// arguments, the per-format digit layout and the staging of x as exact
// integer digits.  The arithmetic is described at the top of qgemv_tma.cu.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "qformat.cuh"

namespace smoe {

constexpr int QG_MAX_EXPERTS = 64;

struct QGArgs {
    const uint8_t *codes[2][QG_MAX_EXPERTS];
    const float *scales[2][QG_MAX_EXPERTS];
    const float *x[QG_MAX_EXPERTS];
    float *y[QG_MAX_EXPERTS];
    unsigned *status;      // device status word (bounded waits)
    int ctas_per_expert;
    int units;             // output rows per expert
    int K;
    int group;
    int scales_tma;        // scales travel with the codes (ngroups % 4 == 0)
    int ns;                // ring slots per warp
    uint32_t stage_bytes;  // bytes of one slot
    uint32_t off_info, off_gmax, off_bars, off_slots;  // shared-memory offsets
    uint32_t off_part;     // row-split kernel: partial row sums
};

template <int BITS>
struct DigitFmt;

template <>
struct DigitFmt<4> {
    static constexpr int NCLASS = 2;     // byte classes per code word
    static constexpr int XSTRIDE = 112;  // digit bytes per chunk (96 + 16 pad: conflict-free)
    static constexpr int CODES_PER_CHUNK = 32;
    static constexpr int WORD_COLS = 8;
    static constexpr float ZINV = 1.0f / 7.5f;
    // class 0: codes of the even columns, class 1: 16 x the codes of the odd
    // columns (the high nibbles, masked in place), one per byte.  The digits
    // of class k are those of x scaled by 2^-SHIFT(k), so the byte products
    // carry the same weight in both classes.
    static __device__ __forceinline__ uint32_t cls(uint32_t w, int k)
    {
        return w & (k == 0 ? 0x0F0F0F0Fu : 0xF0F0F0F0u);
    }
    static constexpr int SHIFT(int k) { return 4 * k; }
    // column (0..7 inside the word) whose digit goes to byte b of class k
    static __device__ __forceinline__ int col(int k, int b) { return 2 * b + k; }
};

template <>
struct DigitFmt<2> {
    static constexpr int NCLASS = 4;
    static constexpr int XSTRIDE = 208;  // 192 + 16 pad
    static constexpr int CODES_PER_CHUNK = 64;
    static constexpr int WORD_COLS = 16;
    static constexpr float ZINV = 1.0f / 1.5f;
    static __device__ __forceinline__ uint32_t cls(uint32_t w, int k)
    {
        return (w >> (2 * k)) & 0x03030303u;
    }
    static constexpr int SHIFT(int) { return 0; }
    static __device__ __forceinline__ int col(int k, int b) { return 4 * b + k; }
};

__device__ __forceinline__ uint4 lds128u(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// c + sum of the four byte products a_i * b_i, a's bytes unsigned (codes,
// possibly shifted into the high nibble), b's bytes signed (x digits).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Balanced base-256 digits of v (|v| <= 2^22): v = d0 + 256 d1 + 65536 d2,
// every digit in [-128, 127].
__device__ __forceinline__ void digits3(int v, int &d0, int &d1, int &d2)
{
    d0 = static_cast<int>(static_cast<signed char>(v & 0xFF));
    const int r = (v - d0) >> 8;
    d1 = static_cast<int>(static_cast<signed char>(r & 0xFF));
    d2 = (r - d1) >> 8;
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// Stages x[0..K) as digits: chunk c occupies XSTRIDE bytes at c*XSTRIDE;
// inside it, the uint4 at (3k + j)*16 holds digit j of byte class k for the
// chunk's 4 code words (word v in component v).  info[c] = {q, q*Sxq, group
// index, 0}.  Called by all threads of the block (blockDim.x % 32 == 0); the
// caller synchronises the block before reading the result.
// Thread t of each pass handles word t of x.  When a group spans a power of
// two of at most 32 words, its words lie in consecutive lanes of one warp and
// the group maximum is a shuffle reduction over values already in registers
// (one read of x, no block barrier); otherwise a first pass gathers the group
// maxima in shared memory with atomics.
// COHERENT: x was written by other CTAs of the running grid (read through L2
// only, never through the read-only path).
template <int BITS, bool COHERENT = false>
__device__ void stage_x_digits(const float *__restrict__ x, int K, int group, uint8_t *smem, uint32_t off_info,
                               uint32_t off_gmax)
{
    using D = DigitFmt<BITS>;
    const int nwords = K / D::WORD_COLS;
    const int gw = group / D::WORD_COLS;  // words per group
    const bool in_warp = gw <= 32 && (gw & (gw - 1)) == 0;
    unsigned *gmax = reinterpret_cast<unsigned *>(smem + off_gmax);
    float4 *info = reinterpret_cast<float4 *>(smem + off_info);

    // largest |x| of a word, +inf when any entry is not finite
    auto word_max = [](const float (&f)[D::WORD_COLS]) {
        float m = 0.f;
        bool finite = true;
#pragma unroll
        for (int i = 0; i < D::WORD_COLS; ++i) {
            m = fmaxf(m, fabsf(f[i]));
            finite = finite && isfinite(f[i]);
        }
        return finite ? m : __uint_as_float(0x7F800000u);
    };
    auto load_word = [&](int v, float (&f)[D::WORD_COLS]) {
        const float4 *p = reinterpret_cast<const float4 *>(x + static_cast<size_t>(v) * D::WORD_COLS);
#pragma unroll
        for (int i = 0; i < D::WORD_COLS / 4; ++i) {
            const float4 q = COHERENT ? __ldcg(p + i) : p[i];
            f[4 * i + 0] = q.x;
            f[4 * i + 1] = q.y;
            f[4 * i + 2] = q.z;
            f[4 * i + 3] = q.w;
        }
    };

    if (!in_warp) {
        const int ngroups = K / group;
        for (int g = threadIdx.x; g < ngroups; g += blockDim.x) gmax[g] = 0u;
        __syncthreads();
        for (int v = threadIdx.x; v < nwords; v += blockDim.x) {
            float f[D::WORD_COLS];
            load_word(v, f);
            atomicMax(&gmax[(v * D::WORD_COLS) / group], __float_as_uint(word_max(f)));
        }
        __syncthreads();
    }
    for (int base = 0; base < nwords; base += blockDim.x) {
        const int v = base + threadIdx.x;
        const bool valid = v < nwords;
        float f[D::WORD_COLS];
        if (valid) {
            load_word(v, f);
        } else {
#pragma unroll
            for (int i = 0; i < D::WORD_COLS; ++i) f[i] = 0.f;
        }
        const int g = valid ? (v * D::WORD_COLS) / group : 0;
        unsigned mb;
        if (in_warp) {
            // a group's gw words are gw consecutive lanes (base is a
            // multiple of 32 and groups are aligned to gw words)
            float m = word_max(f);
            for (int off = 1; off < gw; off <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, off));
            mb = __float_as_uint(m);
        } else {
            mb = valid ? gmax[g] : 0u;
        }
        int S = 0;
        float q = 1.f;
        if (valid) {
            int e = static_cast<int>(mb >> 23) - 127;
            if (e < -105) e = -105;
            const bool finite = mb < 0x7F800000u;
            const float scale = finite ? __uint_as_float(static_cast<unsigned>(127 + 21 - e) << 23) : 0.f;
            q = finite ? __uint_as_float(static_cast<unsigned>(127 + e - 21) << 23) : __uint_as_float(0x7FC00000u);
            // column i of the word is in byte class i % NCLASS; class k is
            // rounded at 2^SHIFT(k) times the step q
            int xq[D::WORD_COLS];
#pragma unroll
            for (int i = 0; i < D::WORD_COLS; ++i) {
                const float sk = scale * __uint_as_float(static_cast<unsigned>(127 - D::SHIFT(i % D::NCLASS)) << 23);
                xq[i] = finite ? __float2int_rn(f[i] * sk) : 0;
            }
            int d[3][D::WORD_COLS];
#pragma unroll
            for (int i = 0; i < D::WORD_COLS; ++i) {
                digits3(xq[i], d[0][i], d[1][i], d[2][i]);
                S += xq[i] * (1 << D::SHIFT(i % D::NCLASS));
            }
            uint8_t *chunk = smem + static_cast<size_t>(v >> 2) * D::XSTRIDE + (v & 3) * 4;
#pragma unroll
            for (int k = 0; k < D::NCLASS; ++k)
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    *reinterpret_cast<uint32_t *>(chunk + (3 * k + j) * 16) =
                        pack4(d[j][D::col(k, 0)], d[j][D::col(k, 1)], d[j][D::col(k, 2)], d[j][D::col(k, 3)]);
        }
        S += __shfl_xor_sync(FULL_MASK, S, 1);
        S += __shfl_xor_sync(FULL_MASK, S, 2);
        if (valid && (v & 3) == 0) info[v >> 2] = make_float4(q, static_cast<float>(S) * q, __int_as_float(g), 0.f);
    }
}


using QGKernelFn = void (*)(QGArgs);

// The register-digit kernel for (bits, nmat, L lanes per row, cpl chunks
// per lane, rpt rows per team), or nullptr when none is built for them.
QGKernelFn qgemv_reg_kernel(int bits, int nmat, int L, int cpl, int rpt);

// The register-digit kernel with every row split into h parts over as many
// classes of warps (512 threads; L = 32, one row per stage), or nullptr.
QGKernelFn qgemv_reg_split_kernel(int bits, int nmat, int cpl, int h);

// Chunks per lane the register-digit kernel takes at most: its digits use
// cpl * 12 * NCLASS registers per thread.
constexpr int reg_kernel_max_cpl(int bits) { return bits == 4 ? 4 : 2; }

}  // namespace smoe
