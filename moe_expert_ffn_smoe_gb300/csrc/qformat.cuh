// Packed Q4/Q2 code format and the affine-dequant fold, device side.
//
// Format (S-MoE "Metal Compute Kernels", sections "Fused FFN Kernels -- One
// Simdgroup Per Output Row" and "Layout assumptions the kernels rely on"):
// one 16-byte chunk of a packed row holds 32 Q4 codes or 64 Q2 codes; inside
// each 32-bit word the code of the lowest column sits in the lowest bits
// (Q4: nibble i of the word is column i; Q2: bit pair i is column i).
//
// Fold.  With w = (c - Z) s / Z, the dot of one group is
//     sum w x = s * (C / Z - Sx),   C = sum c x,  Sx = sum x.
// The kernels never convert a code with an int->float instruction: a code c
// of b bits is OR-ed into the top mantissa bits of 1.0f, giving the exact
// float f = 1 + c / 2^b (2^b = 16 for Q4, 4 for Q2).  The inner loop is then
// a plain FMA chain P = sum f x = Sx + C / 2^b, and per chunk
//     s * (C / Z - Sx) = s * (A * P - (A + 1) * Sx),   A = 2^b / Z,
// so each output row keeps two sums, acc1 = sum s*P and acc2 = sum s*Sx,
// and finishes with A * acc1 - (A + 1) * acc2.  Sx is computed once per
// chunk of x and shared by every row.
#pragma once

#include <stdint.h>

namespace smoe {

template <int BITS>
struct QFmt;

template <>
struct QFmt<4> {
    static constexpr int CODES_PER_CHUNK = 32;  // 16 bytes
    static constexpr int CODES_PER_WORD = 8;
    static constexpr int F4_PER_CHUNK = 8;       // float4s of x under one chunk
    static constexpr int SWZ = 3;                // log2(F4_PER_CHUNK)
    static constexpr float A = 16.0f / 7.5f;     // 2^b / Z
};

template <>
struct QFmt<2> {
    static constexpr int CODES_PER_CHUNK = 64;
    static constexpr int CODES_PER_WORD = 16;
    static constexpr int F4_PER_CHUNK = 16;
    static constexpr int SWZ = 4;
    static constexpr float A = 4.0f / 1.5f;
};

// f = 1 + c / 2^b for the code of column i (0-based) of a 32-bit word.
// Called with a compile-time i in unrolled loops, so the shift is an
// immediate and the mask/OR fold into one LOP3.
template <int BITS>
__device__ __forceinline__ float code_as_f32(uint32_t w, int i)
{
    if (BITS == 4) {
        const int pos = 4 * i;  // nibble bits pos .. pos+3 -> mantissa bits 19..22
        uint32_t t = (pos <= 19) ? (w << (19 - pos)) : (w >> (pos - 19));
        return __uint_as_float((t & 0x00780000u) | 0x3F800000u);
    } else {
        const int pos = 2 * i;  // bit pair pos, pos+1 -> mantissa bits 21..22
        uint32_t t = (pos <= 21) ? (w << (21 - pos)) : (w >> (pos - 21));
        return __uint_as_float((t & 0x00600000u) | 0x3F800000u);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Physical float4 slot of logical float4 q of x in shared memory.  The XOR
// spreads the lanes of a warp, which read the same offset of different
// chunks, over all eight 16-byte bank groups.  Only bits 0..2 change, and
// the mask comes from higher bits, so the map is a bijection inside every
// aligned block of eight float4s.
template <int SWZ>
__device__ __forceinline__ int x_slot(int q)
{
    return q ^ ((q >> SWZ) & 7);
}

// Stages x[0..K) (f32, 16-byte aligned, K a multiple of 4*F4_PER_CHUNK) into
// shared memory with the swizzle above, and writes the sum of each chunk's
// x values into sx[K / CODES_PER_CHUNK].  All threads of the block must call
// it; blockDim.x must be a multiple of 32.
template <int BITS>
__device__ __forceinline__ void stage_x_chunks(const float *__restrict__ x, int K, float4 *xs,
                                               float *sx)
{
    using F = QFmt<BITS>;
    const int nq = K >> 2;
    for (int base = 0; base < nq; base += blockDim.x) {
        const int q = base + threadIdx.x;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q < nq) {
            v = reinterpret_cast<const float4 *>(x)[q];
            xs[x_slot<F::SWZ>(q)] = v;
        }
        float s = (v.x + v.y) + (v.z + v.w);
#pragma unroll
        for (int o = 1; o < F::F4_PER_CHUNK; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (q < nq && (q & (F::F4_PER_CHUNK - 1)) == 0) sx[q >> F::SWZ] = s;
    }
}

}  // namespace smoe
