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
    // Routed launches (route != nullptr): slot e's weights are entry route[e]
    // of device tables of n_route pointers, read after griddepcontrol.wait
    // (the indices come from the previous kernel); codes/scales are unused.
    const uint8_t *const *route_codes[2];
    const float *const *route_scales[2];
    const int *route;
    int n_route;
    unsigned *status;      // device status word (bounded waits)
    int ctas_per_expert;
    int units;             // output rows per expert
    int K;
    int group;
    int scales_tma;        // scales travel with the codes (ngroups % 4 == 0)
    int ns;                // ring slots per warp
    uint32_t stage_bytes;  // bytes of one slot
    uint32_t off_info, off_bars, off_slots;  // shared-memory offsets
    uint32_t off_part;     // row-split kernel: partial row sums
};

template <int BITS>
struct DigitFmt;

// Per format: the byte classes of a code word, the digit layout of a chunk,
// and the centring of the integer dot.  A chunk's integer dot is taken on
// the codes minus OFF (the integer nearest above Z), which keeps it inside
// int32 for every legal x: sum (c - OFF) xq = C - OFF * Sxq.  The chunk's
// contribution to the row is then
//     s q (C / Z - Sxq) = s (q / Z * (C - OFF Sxq) + q Sxq (OFF - Z) / Z),
// so FOLD = (OFF - Z) / Z multiplies q * Sxq.
template <>
struct DigitFmt<4> {
    static constexpr int NCLASS = 2;     // byte classes per code word
    static constexpr int XSTRIDE = 112;  // digit bytes per chunk (96 + 16 pad: conflict-free)
    static constexpr int CODES_PER_CHUNK = 32;
    static constexpr int WORD_COLS = 8;
    static constexpr float ZINV = 1.0f / 7.5f;
    static constexpr int OFF = 8;
    static constexpr float FOLD = 1.0f / 15.0f;  // (8 - 7.5) / 7.5
    // class 0: the codes of the even columns (low nibbles), class 1: the
    // codes of the odd columns (high nibbles moved down), one per byte, so
    // both classes pair with digits of x on the same grid.
    static __device__ __forceinline__ uint32_t cls(uint32_t w, int k)
    {
        return (k == 0 ? w : (w >> 4)) & 0x0F0F0F0Fu;
    }
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
    static constexpr int OFF = 2;
    static constexpr float FOLD = 1.0f / 3.0f;  // (2 - 1.5) / 1.5
    static __device__ __forceinline__ uint32_t cls(uint32_t w, int k)
    {
        return (w >> (2 * k)) & 0x03030303u;
    }
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

// Balanced base-256 digits of v (|v| <= XQ_MAX): v = d0 + 256 d1 + 65536 d2,
// every digit in [-128, 127].
__device__ __forceinline__ void digits3(int v, int &d0, int &d1, int &d2)
{
    d0 = static_cast<int>(static_cast<signed char>(v & 0xFF));
    const int r = (v - d0) >> 8;
    d1 = static_cast<int>(static_cast<signed char>(r & 0xFF));
    d2 = (r - d1) >> 8;
}

// Largest magnitude three balanced base-256 digits hold: 127 * (1 + 256 + 65536).
constexpr int XQ_MAX = 8355711;

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// c + the exact integer dot of one 16-byte chunk of codes (row word v in
// component v of cw) with the digits dg[3 * NCLASS] of its x, returned as
// sum over classes and planes of 256^j * dp4a(class, digit plane j),
// i.e. c + sum code * xq, in arithmetic modulo 2^32.  Starting from
// c = -OFF * Sxq, the result is the chunk's sum (code - OFF) * xq, which
// fits in int32, so the wrap-around of the intermediate sums is harmless.
template <int BITS>
__device__ __forceinline__ int chunk_dot(const uint4 &cw, const uint4 *dg, int c)
{
    using D = DigitFmt<BITS>;
    int A0 = c, A1 = 0, A2 = 0;
#pragma unroll
    for (int cl = 0; cl < D::NCLASS; ++cl)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t cb = D::cls(word_of(cw, v), cl);
            A0 = dp4a_us(cb, word_of(dg[3 * cl + 0], v), A0);
            A1 = dp4a_us(cb, word_of(dg[3 * cl + 1], v), A1);
            A2 = dp4a_us(cb, word_of(dg[3 * cl + 2], v), A2);
        }
    const uint32_t C = static_cast<uint32_t>(A2) * 65536u + static_cast<uint32_t>(A1) * 256u + static_cast<uint32_t>(A0);
    return static_cast<int>(C);
}

// Stages x[0..K) as digits: chunk c occupies XSTRIDE bytes at c*XSTRIDE;
// inside it, the uint4 at (3k + j)*16 holds digit j of byte class k for the
// chunk's 4 code words (word v in component v).  info[c] = {q, q * Sxq *
// FOLD, group index, -OFF * Sxq (int bits)}.  Called by all threads of the
// block (blockDim.x % 32 == 0), or by one whole warp; the caller
// synchronises them before reading the result.
//
// Rounding grid.  Each 16-byte chunk of codes (32 Q4 or 64 Q2 columns) has
// its own power-of-two step q, the smallest for which the chunk's largest
// |x| rounds to at most XQ_MAX steps: that largest |x| is then at least
// 4177856 q, and every x of the chunk is xq * q + r with |r| <= q / 2.
// Thread t of each pass handles word t of x, so a chunk's four words are
// four consecutive lanes and its maximum is two shuffles.
// COHERENT: x was written by other CTAs of the running grid (read through L2
// only, never through the read-only path).
// tid / nthreads: this thread's index among the threads that stage (all of
// the block by default, or one warp: lane and 32); nthreads % 32 == 0.
template <int BITS, bool COHERENT = false>
__device__ void stage_x_digits(const float *__restrict__ x, int K, int group, uint8_t *smem, uint32_t off_info,
                               int tid = -1, int nthreads = 0)
{
    if (tid < 0) {
        tid = static_cast<int>(threadIdx.x);
        nthreads = static_cast<int>(blockDim.x);
    }
    using D = DigitFmt<BITS>;
    const int nwords = K / D::WORD_COLS;  // a multiple of 4: K is a multiple of the chunk
    float4 *info = reinterpret_cast<float4 *>(smem + off_info);

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

    // the words of the next pass are loaded before the current one is
    // converted, so the passes' loads overlap (one warp staging a vector
    // takes several passes)
    float fn[D::WORD_COLS];
    if (tid < nwords) load_word(tid, fn);
    for (int base = 0; base < nwords; base += nthreads) {
        const int v = base + tid;
        const bool valid = v < nwords;
        float f[D::WORD_COLS];
#pragma unroll
        for (int i = 0; i < D::WORD_COLS; ++i) f[i] = valid ? fn[i] : 0.f;
        if (v + nthreads < nwords) load_word(v + nthreads, fn);
        // largest |x| of the chunk, +inf when any entry is not finite
        float m = 0.f;
        bool finite = true;
#pragma unroll
        for (int i = 0; i < D::WORD_COLS; ++i) {
            m = fmaxf(m, fabsf(f[i]));
            finite = finite && isfinite(f[i]);
        }
        if (!finite) m = __uint_as_float(0x7F800000u);
        m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, 1));
        m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, 2));
        const unsigned mb = __float_as_uint(m);
        const int g = valid ? (v * D::WORD_COLS) / group : 0;
        int S = 0;
        float q = 1.f;
        if (valid) {
            // e = floor(log2 max|x|), at least -104 so that q stays a normal float
            int e = static_cast<int>(mb >> 23) - 127;
            if (e < -104) e = -104;
            const bool fin = mb < 0x7F800000u;
            // scale = 1 / q = 2^(22 - e) puts max|x| in [2^22, 2^23); one
            // step coarser when it would round above XQ_MAX
            float scale = __uint_as_float(static_cast<unsigned>(127 + 22 - e) << 23);
            if (m * scale > static_cast<float>(XQ_MAX)) {
                scale *= 0.5f;
                ++e;
            }
            q = fin ? __uint_as_float(static_cast<unsigned>(127 + e - 22) << 23) : __uint_as_float(0x7FC00000u);
            int xq[D::WORD_COLS];
#pragma unroll
            for (int i = 0; i < D::WORD_COLS; ++i) xq[i] = fin ? __float2int_rn(f[i] * scale) : 0;
            int d[3][D::WORD_COLS];
#pragma unroll
            for (int i = 0; i < D::WORD_COLS; ++i) {
                digits3(xq[i], d[0][i], d[1][i], d[2][i]);
                S += xq[i];
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
        if (valid && (v & 3) == 0) {
            // |S| <= 64 XQ_MAX, so OFF * S fits in int32
            const int negoff = static_cast<int>(0u - static_cast<uint32_t>(D::OFF) * static_cast<uint32_t>(S));
            info[v >> 2] = make_float4(q, static_cast<float>(S) * q * D::FOLD, __int_as_float(g), __int_as_float(negoff));
        }
    }
}


// The weights of slot e: the launch's own pointers, or for a routed launch
// (called after griddepcontrol.wait) the table entries of expert route[e].
// Returns false for a routed index outside [0, n_route) or a table entry
// that is null or not 16-byte aligned; the caller then records
// kStatusRoute and writes NaN to the slot's outputs.
__device__ __forceinline__ bool slot_weights(const QGArgs &a, int e, int nmat, const uint8_t *(&c)[2],
                                             const float *(&s)[2])
{
    if (!a.route) {
        c[0] = a.codes[0][e];
        c[1] = a.codes[nmat - 1][e];
        s[0] = a.scales[0][e];
        s[1] = a.scales[nmat - 1][e];
        return true;
    }
    const int idx = a.route[e];
    if (idx < 0 || idx >= a.n_route) return false;
    c[0] = a.route_codes[0][idx];
    c[1] = a.route_codes[nmat - 1][idx];
    s[0] = a.route_scales[0][idx];
    s[1] = a.route_scales[nmat - 1][idx];
    // the bulk copies need 16-byte aligned sources: a table entry that is
    // null or misaligned is refused like a bad index, before any copy
    const uintptr_t bad = (reinterpret_cast<uintptr_t>(c[0]) | reinterpret_cast<uintptr_t>(c[1]) |
                           reinterpret_cast<uintptr_t>(s[0]) | reinterpret_cast<uintptr_t>(s[1])) & 15u;
    return bad == 0 && c[0] && c[1] && s[0] && s[1];
}

// Every thread of the block: NaN into y[r0, r1) (a routed slot whose index
// is out of range), and one thread records the status.
__device__ __forceinline__ void fail_route(const QGArgs &a, float *y, int r0, int r1)
{
    for (int i = r0 + static_cast<int>(threadIdx.x); i < r1; i += blockDim.x) y[i] = __uint_as_float(0x7FC00000u);
    if (threadIdx.x == 0 && a.status) atomicExch(a.status, kStatusRoute);
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
