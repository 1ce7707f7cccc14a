// Decode GEMV with the token's digits held in registers.
//
// Same operations and the same exact integer arithmetic as qgemv_tma.cu
// (S-MoE page "Metal Compute Kernels", section "Fused FFN Kernels -- One
// Simdgroup Per Output Row"; w = (code - Z) s / Z, folded per group), for
// row lengths where every lane of a team can keep the x digits of all the
// chunks it ever touches in registers (regdot.cuh).  The inner loop reads
// only codes and one scale per chunk from shared memory: the scales of a
// stage travel with its codes (the kernel is used only when a row's scales
// are a multiple of 16 bytes, i.e. groups per row % 4 == 0).
// Streaming is as in qgemv_tma.cu: every warp owns a ring of `ns`
// shared-memory slots filled by cp.async.bulk and waits only on its own.
// The bulk copies of a stage are issued by up to four lanes at once (codes
// and scales of each matrix).
//
// Row split (H > 1): every row is cut into H parts of K / H columns; part h
// of row i is "virtual row" i H + h, so a matrix reads as H times as many
// rows of K / H columns with the same bytes in the same places.  Warp w
// only ever streams virtual rows with h = w % H (one row per stage, NW a
// multiple of H), so its lanes hold the digits of 1 / H of x: the CTA runs
// 16 warps instead of 12.  Parts of a row are summed in shared memory after
// the last stage, then SiLU(gate) * up is applied.
#include "regdot.cuh"

namespace smoe {

namespace {

template <int BITS, int NMAT, int L, int CPL, int RPT, int H>
__global__ void __launch_bounds__(H == 1 ? 384 : 512, 1) qgemv_reg(const __grid_constant__ QGArgs a)
{
    static_assert(H == 1 || (L == 32 && RPT == 1), "row split streams one row per stage");
    using RD = RegDot<BITS, NMAT, L, CPL, RPT>;
    constexpr int TEAMS = RD::TEAMS;
    constexpr int R = RD::R;                   // rows of each matrix per stage
    constexpr uint32_t ROW_BYTES = RD::ROW_BYTES;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int NW = blockDim.x >> 5;
    const int e = blockIdx.x / a.ctas_per_expert;
    const int bi = blockIdx.x - e * a.ctas_per_expert;
    const int r0 = static_cast<int>(static_cast<long long>(a.units) * bi / a.ctas_per_expert);
    const int r1 = static_cast<int>(static_cast<long long>(a.units) * (bi + 1) / a.ctas_per_expert);
    const int u0 = r0 * H, u1 = r1 * H;  // virtual rows (H == 1: the rows)
    const int nst = (u1 - u0 + R - 1) / R;
    const int my = warp < nst ? (nst - warp + NW - 1) / NW : 0;  // stages of this warp
    const int ngroups = a.K / a.group / H;  // groups of a virtual row
    const int ns = a.ns;
    const uint32_t bars = sbase + a.off_bars + static_cast<uint32_t>(warp * ns) * 8u;
    const uint32_t slots = sbase + a.off_slots + static_cast<uint32_t>(warp * ns) * a.stage_bytes;
    const uint32_t scales_off = static_cast<uint32_t>(NMAT * R) * ROW_BYTES;
    const uint32_t sbytes_row = static_cast<uint32_t>(ngroups) * 4u;  // scales travel with the codes
    float *part = reinterpret_cast<float *>(smem + a.off_part);    // H > 1: [u1 - u0][NMAT]

    // Copy roles: lanes 0..NMAT-1 the codes of matrix `lane`, lanes
    // NMAT..2 NMAT-1 the scales of matrix `lane - NMAT`.  src0 is this lane's source for the warp's first
    // stage; each later stage of the warp is NW * R rows further on.
    const int role_m = lane < NMAT ? lane : lane - NMAT;
    const bool role_codes = lane < NMAT;
    const bool role_any = lane < 2 * NMAT;
    const uint8_t *src0 = nullptr;
    size_t src_step = 0;
    uint32_t row_b = 0, dst_off = 0;
    auto set_sources = [&](const uint8_t *const (&cm)[2], const float *const (&sm)[2]) {
        if (!role_any) return;
        const int m = role_m < NMAT ? role_m : 0;
        const size_t first_row = static_cast<size_t>(u0) + static_cast<size_t>(warp) * R;
        if (role_codes) {
            src0 = cm[m] + first_row * ROW_BYTES;
            row_b = ROW_BYTES;
            dst_off = static_cast<uint32_t>(m * R) * ROW_BYTES;
        } else {
            src0 = reinterpret_cast<const uint8_t *>(sm[m] + first_row * ngroups);
            row_b = sbytes_row;
            dst_off = scales_off + static_cast<uint32_t>(m * R) * sbytes_row;
        }
        src_step = static_cast<size_t>(NW) * R * row_b;
    };

    // The whole warp: the copies of its k-th stage into slot `si`.
    auto issue = [&](int k, int si) {
        const int us = u0 + (warp + k * NW) * R;
        const uint32_t n = static_cast<uint32_t>(min(R, u1 - us));
        const uint32_t slot = slots + static_cast<uint32_t>(si) * a.stage_bytes;
        const uint32_t bar = bars + static_cast<uint32_t>(si) * 8u;
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NMAT) * n * (ROW_BYTES + sbytes_row));
        __syncwarp();
        if (role_any) bulk_g2s(slot + dst_off, src0 + static_cast<size_t>(k) * src_step, n * row_b, bar);
    };

    if (lane == 0) {
        for (int i = 0; i < ns; ++i) mbar_init(bars + 8u * i, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // Weights never depend on an earlier kernel: the first stage goes out
    // before waiting for it (unless the weights themselves are chosen by the
    // previous kernel: a routed launch), and for the down projection (one
    // row per stage) the second one too.  The rest of the first wave
    // follows the staging of x, whose loads would otherwise queue behind it.
    // (Measured in the 8-expert step: two early stages for down took the
    // step from 19.62 to 19.53 us; more early copies, or early copies of
    // gate/up, slow the previous kernel's last CTAs, which set the step's
    // critical path.)
    const int first = my < ns ? my : ns;
    const int early = (!a.route && NMAT == 1 && first > 1) ? 2 : 1;
    const uint8_t *wc[2];
    const float *ws[2];
    if (!a.route) {
        slot_weights(a, e, NMAT, wc, ws);
        set_sources(wc, ws);
        for (int k = 0; k < early && k < first; ++k) issue(k, k);
    }

    pdl_wait();
    if (a.route) {
        if (!slot_weights(a, e, NMAT, wc, ws)) {
            fail_route(a, a.y[e], r0, r1);
            return;
        }
        set_sources(wc, ws);
        if (first > 0) issue(0, 0);
    }
    stage_x_digits<BITS>(a.x[e], a.K, a.group, smem, a.off_info);
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    for (int k = a.route ? 1 : early; k < first; ++k) issue(k, k);

    const int team = lane / L;
    const int u = lane % L;

    // This lane's digits, q / Z, q * Sxq and scale offsets, for good.
    RD rd;
    const int h = H == 1 ? 0 : warp % H;
    rd.load(sbase, a.off_info, u, h * RD::KC, h * ngroups);

    int k = 0, si = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (; k < my; ++k) {
        ok = mbar_wait_bounded(bars + static_cast<uint32_t>(si) * 8u, phase, a.status, 1u);
        ok = __all_sync(FULL_MASK, ok);
        if (!ok) break;
        const uint32_t slot = slots + static_cast<uint32_t>(si) * a.stage_bytes;
        const int us = u0 + (warp + k * NW) * R;
        float acc[NMAT][RPT];
        rd.stage(slot, team, u, sbytes_row, acc);
        __syncwarp();
        if (k + ns < my) {
            fence_proxy_async_smem();
            issue(k + ns, si);
        }
        if (u == 0) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int ul = r * TEAMS + team;
                if (us + ul < u1) {
                    if (H > 1) {
#pragma unroll
                        for (int m = 0; m < NMAT; ++m) part[(us + ul - u0) * NMAT + m] = acc[m][r];
                    } else {
                        float out = acc[0][r];
                        if (NMAT == 2) out = silu_f32(acc[0][r]) * acc[NMAT - 1][r];
                        a.y[e][us + ul] = out;
                    }
                }
            }
        }
        if (++si == ns) {
            si = 0;
            phase ^= 1u;
        }
    }
    if (!ok && lane == 0) {
        // A copy never completed: wait (bounded) for the ones still in
        // flight (stages k .. min(k + ns, my) - 1, in ring order from si)
        // before the CTA's shared memory is released.
        const int last = (k + ns < my) ? k + ns : my;
        for (int kk = k; kk < last; ++kk) {
            mbar_wait_bounded(bars + static_cast<uint32_t>(si) * 8u, phase, nullptr, 0u);
            if (++si == ns) {
                si = 0;
                phase ^= 1u;
            }
        }
    }
    if (H > 1) {
        // every warp has stored its parts (a warp that gave up left garbage
        // and recorded the failure): add the parts of each row
        __syncthreads();
        for (int i = threadIdx.x; i < r1 - r0; i += blockDim.x) {
            float v[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                v[m] = 0.f;
#pragma unroll
                for (int p = 0; p < H; ++p) v[m] += part[(i * H + p) * NMAT + m];
            }
            a.y[e][r0 + i] = NMAT == 2 ? silu_f32(v[0]) * v[NMAT - 1] : v[0];
        }
    }
}

template <int BITS, int NMAT, int L, int RPT>
QGKernelFn pick_cpl(int cpl)
{
    switch (cpl) {
    case 1: return qgemv_reg<BITS, NMAT, L, 1, RPT, 1>;
    case 2: return qgemv_reg<BITS, NMAT, L, 2, RPT, 1>;
    case 3: return BITS == 4 ? qgemv_reg<BITS, NMAT, L, (BITS == 4 ? 3 : 1), RPT, 1> : nullptr;
    case 4: return BITS == 4 ? qgemv_reg<BITS, NMAT, L, (BITS == 4 ? 4 : 1), RPT, 1> : nullptr;
    default: return nullptr;
    }
}

template <int BITS, int NMAT, int RPT>
QGKernelFn pick_l(int L, int cpl)
{
    if (L == 32) return pick_cpl<BITS, NMAT, 32, RPT>(cpl);
    if (L == 16) return pick_cpl<BITS, NMAT, 16, RPT>(cpl);
    if (L == 8) return pick_cpl<BITS, NMAT, 8, RPT>(cpl);
    return nullptr;
}

}  // namespace

QGKernelFn qgemv_reg_split_kernel(int bits, int nmat, int cpl, int h)
{
    // built for gate/up: Q4 with 1 or 2 chunks per lane, Q2 with 1
    if (nmat != 2 || (h != 2 && h != 4)) return nullptr;
    if (bits == 4) {
        if (cpl == 1) return h == 2 ? qgemv_reg<4, 2, 32, 1, 1, 2> : qgemv_reg<4, 2, 32, 1, 1, 4>;
        if (cpl == 2) return h == 2 ? qgemv_reg<4, 2, 32, 2, 1, 2> : qgemv_reg<4, 2, 32, 2, 1, 4>;
        return nullptr;
    }
    if (cpl == 1) return h == 2 ? qgemv_reg<2, 2, 32, 1, 1, 2> : qgemv_reg<2, 2, 32, 1, 1, 4>;
    return nullptr;
}

QGKernelFn qgemv_reg_kernel(int bits, int nmat, int L, int cpl, int rpt)
{
    // gate/up (two matrices) always streams one row per team and stage
    if (nmat == 2) {
        if (rpt != 1) return nullptr;
        return bits == 4 ? pick_l<4, 2, 1>(L, cpl) : pick_l<2, 2, 1>(L, cpl);
    }
    if (rpt == 1) return bits == 4 ? pick_l<4, 1, 1>(L, cpl) : pick_l<2, 1, 1>(L, cpl);
    return nullptr;
}

}  // namespace smoe
