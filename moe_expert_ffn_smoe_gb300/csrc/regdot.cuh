// The lane state and the per-stage dot products of the register-digit decode
// kernels (qgemv_reg.cu, expert_ffn.cu).
//
// Same arithmetic as the S-MoE page "Metal Compute Kernels", section "Fused
// FFN Kernels -- One Simdgroup Per Output Row" (w = (code - Z) s / Z, folded
// per group), rewritten on exact integers (see qgemv_tma.cu):
//  * A team of L lanes covers one row; lane u always handles the 16-byte
//    chunks c = u + j L (j < CPL), so its digits of x, q / Z, q * Sxq and
//    scale offset for those chunks are loaded from the staged x once and
//    kept in registers.
//  * A stage in shared memory holds the codes of NMAT * R rows (R = TEAMS *
//    RPT rows per matrix, ROW_BYTES each) followed by their scales
//    (`sbytes_row` bytes per row).  Row m R + r TEAMS + team of the stage is
//    matrix m's row for team `team`, r-th of its RPT rows.
#pragma once

#include "qgemv_tma.cuh"

namespace smoe {

template <int BITS, int NMAT, int L, int CPL, int RPT>
struct RegDot {
    using D = DigitFmt<BITS>;
    static constexpr int TEAMS = 32 / L;
    static constexpr int R = TEAMS * RPT;          // rows of each matrix per stage
    static constexpr int KC = L * CPL;             // 16-byte code chunks per row
    static constexpr uint32_t ROW_BYTES = KC * 16u;
    static constexpr int ND = 3 * D::NCLASS;       // digit words (uint4) per chunk

    uint4 dg[CPL][ND];
    float qz[CPL], qs[CPL];
    int c0[CPL];
    uint32_t soff[CPL];

    // Lane u's digits, q / Z, q * Sxq * FOLD, -OFF * Sxq and scale byte offsets from x staged at
    // sbase (digits) and sbase + off_info (chunk info).  The rows streamed
    // may be a part of x's length: chunks chunk0 .. chunk0 + KC - 1 of x,
    // whose scales start at group `group0` of the full row.
    __device__ __forceinline__ void load(uint32_t sbase, uint32_t off_info, int u, int chunk0 = 0, int group0 = 0)
    {
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = chunk0 + u + j * L;
            const uint32_t xc = sbase + static_cast<uint32_t>(c) * D::XSTRIDE;
#pragma unroll
            for (int t = 0; t < ND; ++t) dg[j][t] = lds128u(xc + static_cast<uint32_t>(t) * 16u);
            const float4 inf = lds128f(sbase + off_info + static_cast<uint32_t>(c) * 16u);
            qz[j] = inf.x * D::ZINV;
            qs[j] = inf.y;
            c0[j] = __float_as_int(inf.w);
            soff[j] = static_cast<uint32_t>(__float_as_int(inf.z) - group0) * 4u;
        }
    }

    // acc[m][r] = (row m R + r TEAMS + team of the stage in `slot`) . x,
    // summed over the team's L lanes (every lane of the team ends with it).
    __device__ __forceinline__ void stage(uint32_t slot, int team, int u, uint32_t sbytes_row,
                                          float (&acc)[NMAT][RPT]) const
    {
        const uint32_t code_lane = slot + static_cast<uint32_t>(team) * ROW_BYTES + static_cast<uint32_t>(u) * 16u;
        const uint32_t scale_lane =
            slot + static_cast<uint32_t>(NMAT * R) * ROW_BYTES + static_cast<uint32_t>(team) * sbytes_row;
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r) acc[m][r] = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    // row m R + r TEAMS + team, chunk u + j L
                    const uint4 cw = lds128u(code_lane + static_cast<uint32_t>((m * R + r * TEAMS) * ROW_BYTES +
                                                                               j * L * 16));
                    const int C = chunk_dot<BITS>(cw, dg[j], c0[j]);  // sum (code - OFF) * xq
                    const float sc =
                        lds_f32(scale_lane + static_cast<uint32_t>(m * R + r * TEAMS) * sbytes_row + soff[j]);
                    acc[m][r] = fmaf(sc, fmaf(static_cast<float>(C), qz[j], qs[j]), acc[m][r]);
                }
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
                for (int off = L / 2; off > 0; off >>= 1) acc[m][r] += __shfl_xor_sync(FULL_MASK, acc[m][r], off);
    }
};

}  // namespace smoe
