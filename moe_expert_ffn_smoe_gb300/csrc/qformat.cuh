// Packed Q4/Q2 code format and the affine-dequant fold, device side.
//
// Format (S-MoE "Metal Compute Kernels", sections "Fused FFN Kernels -- One
// Simdgroup Per Output Row" and "Layout assumptions the kernels rely on"):
// one 16-byte chunk of a packed row holds 32 Q4 codes or 64 Q2 codes; inside
// each 32-bit word the code of the lowest column sits in the lowest bits
// (Q4: nibble i of the word is column i; Q2: bit pair i is column i).
//
// Weights.  The kernels never convert a code with an int->float
// instruction: a code c of b bits is OR-ed into the top mantissa bits of
// 1.0f, giving the exact float f = 1 + c / 2^b (2^b = 16 for Q4, 4 for Q2),
// and f - (1 + Z / 2^b) = (c - Z) / 2^b is exact too (both are multiples of
// 2^-(b+1) within a factor two of each other).  So the inner loop is a plain
// FMA chain over the exact centred weights, P = sum (c - Z) / 2^b * x, per
// chunk acc += s * P, and the row finishes with A * acc, A = 2^b / Z:
//     sum w x = sum s (c - Z) / Z * x = A * sum s * P.
// No large terms cancel: every product is the weight's own share of the
// dot, so the f32 rounding is relative to sum |w x|.
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
    static constexpr float BIAS = 1.46875f;      // 1 + Z / 2^b
};

template <>
struct QFmt<2> {
    static constexpr int CODES_PER_CHUNK = 64;
    static constexpr int CODES_PER_WORD = 16;
    static constexpr int F4_PER_CHUNK = 16;
    static constexpr int SWZ = 4;
    static constexpr float A = 4.0f / 1.5f;
    static constexpr float BIAS = 1.375f;
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

// (c - Z) / 2^b for the code of column i of a 32-bit word, exact.
template <int BITS>
__device__ __forceinline__ float code_centred(uint32_t w, int i)
{
    return code_as_f32<BITS>(w, i) - QFmt<BITS>::BIAS;
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
// shared memory with the swizzle above.  All threads of the block must call
// it.
template <int BITS>
__device__ __forceinline__ void stage_x_chunks(const float *__restrict__ x, int K, float4 *xs)
{
    using F = QFmt<BITS>;
    const int nq = K >> 2;
    for (int q = threadIdx.x; q < nq; q += blockDim.x) xs[x_slot<F::SWZ>(q)] = reinterpret_cast<const float4 *>(x)[q];
}

}  // namespace smoe
