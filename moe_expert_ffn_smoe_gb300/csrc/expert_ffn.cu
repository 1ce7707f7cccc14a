// The whole routed-expert FFN for one token over n experts in one launch.
//
// Computes, for every expert e (S-MoE page "Metal Compute Kernels", section
// "Fused FFN Kernels -- One Simdgroup Per Output Row", and its "Grouped
// Expert Dispatch", which batches all ready experts into one submission):
//     hidden_e = SiLU(gate_e . x) * (up_e . x)
//     out_e    = down_e . hidden_e
// with the exact integer dot products of regdot.cuh.
//
// Grid: `cpe` CTAs per expert, one per SM.  A CTA owns a row range of its
// expert's gate/up (phase 1) and a row range of its expert's down (phase 2).
// Every warp streams one sequence of stages through its ring of shared-
// memory slots: its phase-1 stages, then its phase-2 stages.  Down weights
// never depend on hidden, so a slot freed in phase 1 is refilled with the
// next stage whichever phase it belongs to: the down weights stream while
// phase 1 finishes and while the CTA waits for its expert's hidden vector.
//
// Between the phases the CTAs of one expert meet on a counter in the
// caller's workspace: each adds one after storing its hidden rows (release),
// then waits (bounded) until all cpe have (acquire) before staging hidden as
// x of phase 2.  The last CTA to pass the wait resets the counters, so a
// completed launch leaves them zero for the next one; a launch that starts
// while the previous one still runs touches them only after
// griddepcontrol.wait, i.e. after that launch has completed.
// The waits need all CTAs of the grid resident together: the grid never
// exceeds one CTA per SM, and it is a cooperative launch, so CUDA starts it
// only when every CTA can be resident (and refuses a grid that never
// could).  A wait that still gives up (about two seconds) records a status
// and skips phase 2; the counters must then be zeroed again by the caller.
#include "regdot.cuh"

namespace smoe {

struct FFNArgs {
    const uint8_t *codes[3][QG_MAX_EXPERTS];  // gate, up, down
    const float *scales[3][QG_MAX_EXPERTS];
    const float *x;        // [d_model], the token, shared by all experts
    float *hidden;         // [n][d_ff] (workspace)
    float *out;            // [n][d_model]
    unsigned *sync;        // [2][QG_MAX_EXPERTS]: arrivals, departures (workspace)
    unsigned *status;      // device status word
    int cpe;               // CTAs per expert
    int d_model, d_ff, group;
    int ns;                // ring slots per warp
    uint32_t slot_bytes;
    uint32_t off_info, off_bars, off_slots;
};

namespace {

template <int BITS, int L1, int CPL1, int L2, int CPL2>
__global__ void __launch_bounds__(384, 1) expert_ffn(const __grid_constant__ FFNArgs a)
{
    using G = RegDot<BITS, 2, L1, CPL1, 1>;   // gate/up: one row pair per team and stage
    using Dn = RegDot<BITS, 1, L2, CPL2, 2>;  // down: two rows per team and stage

    extern __shared__ uint8_t smem_raw[];
    __shared__ int handoff_ok;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int NW = blockDim.x >> 5;
    const int e = blockIdx.x / a.cpe;
    const int bi = blockIdx.x - e * a.cpe;
    // this CTA's rows: [u0, u1) of d_ff (phase 1), [v0, v1) of d_model (phase 2)
    const int u0 = static_cast<int>(static_cast<long long>(a.d_ff) * bi / a.cpe);
    const int u1 = static_cast<int>(static_cast<long long>(a.d_ff) * (bi + 1) / a.cpe);
    const int v0 = static_cast<int>(static_cast<long long>(a.d_model) * bi / a.cpe);
    const int v1 = static_cast<int>(static_cast<long long>(a.d_model) * (bi + 1) / a.cpe);
    const int nst1 = (u1 - u0 + G::R - 1) / G::R;
    const int nst2 = (v1 - v0 + Dn::R - 1) / Dn::R;
    const int my1 = warp < nst1 ? (nst1 - warp + NW - 1) / NW : 0;
    const int my2 = warp < nst2 ? (nst2 - warp + NW - 1) / NW : 0;
    const int nsg = my1 + my2;  // this warp's stages: phase 1, then phase 2
    const uint32_t sb1 = static_cast<uint32_t>(a.d_model / a.group) * 4u;  // scale bytes per gate/up row
    const uint32_t sb2 = static_cast<uint32_t>(a.d_ff / a.group) * 4u;     // scale bytes per down row
    const int ns = a.ns;
    const uint32_t bars = sbase + a.off_bars + static_cast<uint32_t>(warp * ns) * 8u;
    const uint32_t slots = sbase + a.off_slots + static_cast<uint32_t>(warp * ns) * a.slot_bytes;

    // Copy roles.  Phase 1: lanes 0, 1 the codes of gate, up; lanes 2, 3
    // their scales.  Phase 2: lane 0 the down codes, lane 1 their scales.
    // srcN is this lane's source for the warp's first stage of phase N; each
    // later stage is NW * R rows further on.
    const uint8_t *src1 = nullptr, *src2 = nullptr;
    size_t step1 = 0, step2 = 0;
    uint32_t rowb1 = 0, rowb2 = 0, dst1 = 0, dst2 = 0;
    if (lane < 4) {
        const int m = lane & 1;
        const size_t r0 = static_cast<size_t>(u0) + static_cast<size_t>(warp) * G::R;
        if (lane < 2) {
            src1 = a.codes[m][e] + r0 * G::ROW_BYTES;
            rowb1 = G::ROW_BYTES;
            dst1 = static_cast<uint32_t>(m * G::R) * G::ROW_BYTES;
        } else {
            src1 = reinterpret_cast<const uint8_t *>(a.scales[m][e]) + r0 * sb1;
            rowb1 = sb1;
            dst1 = static_cast<uint32_t>(2 * G::R) * G::ROW_BYTES + static_cast<uint32_t>(m * G::R) * sb1;
        }
        step1 = static_cast<size_t>(NW) * G::R * rowb1;
    }
    if (lane < 2) {
        const size_t r0 = static_cast<size_t>(v0) + static_cast<size_t>(warp) * Dn::R;
        if (lane == 0) {
            src2 = a.codes[2][e] + r0 * Dn::ROW_BYTES;
            rowb2 = Dn::ROW_BYTES;
            dst2 = 0u;
        } else {
            src2 = reinterpret_cast<const uint8_t *>(a.scales[2][e]) + r0 * sb2;
            rowb2 = sb2;
            dst2 = static_cast<uint32_t>(Dn::R) * Dn::ROW_BYTES;
        }
        step2 = static_cast<size_t>(NW) * Dn::R * rowb2;
    }

    // The whole warp: the copies of its stage s into slot si.
    auto issue = [&](int s, int si) {
        const uint32_t slot = slots + static_cast<uint32_t>(si) * a.slot_bytes;
        const uint32_t bar = bars + static_cast<uint32_t>(si) * 8u;
        if (s < my1) {
            const int us = u0 + (warp + s * NW) * G::R;
            const uint32_t n = static_cast<uint32_t>(min(G::R, u1 - us));
            if (lane == 0) mbar_arrive_expect_tx(bar, 2u * n * (G::ROW_BYTES + sb1));
            __syncwarp();
            if (lane < 4) bulk_g2s(slot + dst1, src1 + static_cast<size_t>(s) * step1, n * rowb1, bar);
        } else {
            const int k = s - my1;
            const int vs = v0 + (warp + k * NW) * Dn::R;
            const uint32_t n = static_cast<uint32_t>(min(Dn::R, v1 - vs));
            if (lane == 0) mbar_arrive_expect_tx(bar, n * (Dn::ROW_BYTES + sb2));
            __syncwarp();
            if (lane < 2) bulk_g2s(slot + dst2, src2 + static_cast<size_t>(k) * step2, n * rowb2, bar);
        }
    };

    if (lane == 0) {
        for (int i = 0; i < ns; ++i) mbar_init(bars + 8u * i, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int first = nsg < ns ? nsg : ns;
    if (first > 0) issue(0, 0);  // weights never depend on an earlier kernel

    pdl_wait();
    stage_x_digits<BITS>(a.x, a.d_model, a.group, smem, a.off_info);
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    for (int s = 1; s < first; ++s) issue(s, s);

    int s = 0, si = 0;  // next stage to wait for, its slot
    uint32_t phase = 0;
    bool ok = true;
    auto advance = [&]() {
        ++s;
        if (++si == ns) {
            si = 0;
            phase ^= 1u;
        }
    };

    // ---- phase 1: gate/up rows -> hidden
    {
        const int team = lane / L1;
        const int u = lane % L1;
        G g;
        g.load(sbase, a.off_info, u);
        float *hid = a.hidden + static_cast<size_t>(e) * a.d_ff;
        while (s < my1) {
            ok = __all_sync(FULL_MASK, mbar_wait_bounded(bars + static_cast<uint32_t>(si) * 8u, phase, a.status, 1u));
            if (!ok) break;
            float acc[2][1];
            g.stage(slots + static_cast<uint32_t>(si) * a.slot_bytes, team, u, sb1, acc);
            __syncwarp();
            if (s + ns < nsg) {
                fence_proxy_async_smem();
                issue(s + ns, si);
            }
            const int row = u0 + (warp + s * NW) * G::R + team;
            if (u == 0 && row < u1) hid[row] = silu_f32(acc[0][0]) * acc[1][0];
            advance();
        }
    }

    // ---- hand-off: every CTA of expert e has stored its hidden rows.
    // Each thread's stores are made visible device-wide before the barrier;
    // thread 0 then counts the CTA in (release) and waits for the others
    // (acquire); the barrier after it orders every thread's loads of hidden.
    __threadfence();
    ok = __syncthreads_and(ok);
    if (threadIdx.x == 0) {
        int h = 0;
        if (ok) {
            atomicAdd(&a.sync[e], 1u);
            if (wait_count(&a.sync[e], static_cast<unsigned>(a.cpe))) {
                h = 1;
                const unsigned before = atomicAdd(&a.sync[QG_MAX_EXPERTS + e], 1u);
                if (before == static_cast<unsigned>(a.cpe) - 1u) {
                    // every CTA of expert e has passed the wait
                    atomicExch(&a.sync[e], 0u);
                    atomicExch(&a.sync[QG_MAX_EXPERTS + e], 0u);
                }
            } else {
                atomicExch(a.status, 2u);
            }
        }
        handoff_ok = h;
    }
    __syncthreads();
    ok = handoff_ok != 0;

    // ---- phase 2: down rows of hidden_e -> out
    if (ok) {
        stage_x_digits<BITS, true>(a.hidden + static_cast<size_t>(e) * a.d_ff, a.d_ff, a.group, smem, a.off_info);
        __syncthreads();
        const int team = lane / L2;
        const int u = lane % L2;
        Dn d;
        d.load(sbase, a.off_info, u);
        float *out = a.out + static_cast<size_t>(e) * a.d_model;
        while (s < nsg) {
            ok = __all_sync(FULL_MASK, mbar_wait_bounded(bars + static_cast<uint32_t>(si) * 8u, phase, a.status, 1u));
            if (!ok) break;
            float acc[1][2];
            d.stage(slots + static_cast<uint32_t>(si) * a.slot_bytes, team, u, sb2, acc);
            __syncwarp();
            if (s + ns < nsg) {
                fence_proxy_async_smem();
                issue(s + ns, si);
            }
            const int vs = v0 + (warp + (s - my1) * NW) * Dn::R;
            if (u == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = vs + r * Dn::TEAMS + team;
                    if (row < v1) out[row] = acc[0][r];
                }
            }
            advance();
        }
    }

    if (!ok && lane == 0) {
        // Stages s .. min(s + ns, nsg) - 1 may still be in flight: wait for
        // them (bounded) before the CTA's shared memory is released.
        const int last = (s + ns < nsg) ? s + ns : nsg;
        for (int t = s; t < last; ++t) {
            mbar_wait_bounded(bars + static_cast<uint32_t>(si) * 8u, phase, nullptr, 0u);
            if (++si == ns) {
                si = 0;
                phase ^= 1u;
            }
        }
    }
}

using FFNKernel = void (*)(FFNArgs);

// (L, chunks per lane) of a row of `kc` 16-byte chunks, as the decode
// kernels choose them: the largest team that divides the row with at most
// reg_kernel_max_cpl chunks per lane.
bool team_shape(int bits, int kc, int *L, int *cpl)
{
    for (int l = 32; l >= 8; l >>= 1)
        if (kc % l == 0 && kc / l <= reg_kernel_max_cpl(bits)) {
            *L = l;
            *cpl = kc / l;
            return true;
        }
    return false;
}

template <int BITS, int L1, int CPL1>
FFNKernel pick2(int L2, int cpl2)
{
    if (BITS == 4) {
        if (L2 == 32 && cpl2 == 2) return expert_ffn<BITS, L1, CPL1, 32, 2>;
        if (L2 == 32 && cpl2 == 3) return expert_ffn<BITS, L1, CPL1, 32, (BITS == 4 ? 3 : 2)>;
        if (L2 == 32 && cpl2 == 4) return expert_ffn<BITS, L1, CPL1, 32, (BITS == 4 ? 4 : 2)>;
        if (L2 == 16 && cpl2 == 3) return expert_ffn<BITS, L1, CPL1, 16, (BITS == 4 ? 3 : 2)>;
        if (L2 == 8 && cpl2 == 3) return expert_ffn<BITS, L1, CPL1, 8, (BITS == 4 ? 3 : 2)>;
    } else {
        if (L2 == 32 && cpl2 == 2) return expert_ffn<BITS, L1, CPL1, 32, 2>;
    }
    return nullptr;
}

template <int BITS>
FFNKernel pick_ffn(int L1, int cpl1, int L2, int cpl2)
{
    if (BITS == 4) {
        if (L1 == 32 && cpl1 == 2) return pick2<BITS, 32, 2>(L2, cpl2);
        if (L1 == 32 && cpl1 == 3) return pick2<BITS, 32, (BITS == 4 ? 3 : 2)>(L2, cpl2);
        if (L1 == 32 && cpl1 == 4) return pick2<BITS, 32, (BITS == 4 ? 4 : 2)>(L2, cpl2);
        if (L1 == 16 && cpl1 == 3) return pick2<BITS, 16, (BITS == 4 ? 3 : 2)>(L2, cpl2);
        if (L1 == 8 && cpl1 == 3) return pick2<BITS, 8, (BITS == 4 ? 3 : 2)>(L2, cpl2);
    } else {
        if (L1 == 32 && cpl1 == 2) return pick2<BITS, 32, 2>(L2, cpl2);
    }
    return nullptr;
}

uint32_t round16u(uint32_t v) { return (v + 15u) & ~15u; }

constexpr size_t kFFNSmemBudget = 200 * 1024;

}  // namespace

// One launch over n <= QG_MAX_EXPERTS experts, or *unsupported = true (and
// nothing launched) for shapes the fused kernel does not take.
cudaError_t launch_expert_ffn(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                              const uint8_t *const *uc, const float *const *us, const uint8_t *const *dc,
                              const float *const *ds, const float *x, float *hidden, float *out, unsigned *sync,
                              int d_model, int d_ff, int group, cudaStream_t stream, bool *unsupported)
{
    *unsupported = true;
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    if (n < 1 || n > QG_MAX_EXPERTS || n > dev->sm_count) return cudaSuccess;
    const int cpc = bits == 4 ? 32 : 64;  // codes per 16-byte chunk
    if (d_model % cpc || d_ff % cpc || group % cpc) return cudaSuccess;
    const int kc1 = d_model / cpc, kc2 = d_ff / cpc;
    const int ng1 = d_model / group, ng2 = d_ff / group;
    if (ng1 % 4 || ng2 % 4) return cudaSuccess;  // scales travel with the codes
    int L1, cpl1, L2, cpl2;
    if (!team_shape(bits, kc1, &L1, &cpl1) || !team_shape(bits, kc2, &L2, &cpl2)) return cudaSuccess;
    FFNKernel k = bits == 4 ? pick_ffn<4>(L1, cpl1, L2, cpl2) : pick_ffn<2>(L1, cpl1, L2, cpl2);
    if (!k) return cudaSuccess;

    FFNArgs a = {};
    for (int i = 0; i < n; ++i) {
        a.codes[0][i] = gc[i];
        a.codes[1][i] = uc[i];
        a.codes[2][i] = dc[i];
        a.scales[0][i] = gs[i];
        a.scales[1][i] = us[i];
        a.scales[2][i] = ds[i];
    }
    a.x = x;
    a.hidden = hidden;
    a.out = out;
    a.sync = sync;
    a.status = device_status_word();
    a.cpe = dev->sm_count / n;
    a.d_model = d_model;
    a.d_ff = d_ff;
    a.group = group;

    // shared memory: x digits and chunk info sized for the longer of the two
    // row lengths, per-warp barriers, then the rings
    const int kcmax = kc1 > kc2 ? kc1 : kc2;
    const uint32_t xstride = bits == 4 ? DigitFmt<4>::XSTRIDE : DigitFmt<2>::XSTRIDE;
    a.off_info = static_cast<uint32_t>(kcmax) * xstride;
    a.off_bars = a.off_info + static_cast<uint32_t>(kcmax) * 16u;
    const int teams1 = 32 / L1, teams2 = 32 / L2;
    const uint32_t stage1 = 2u * teams1 * (static_cast<uint32_t>(kc1) * 16u + ng1 * 4u);
    const uint32_t stage2 = 2u * teams2 * (static_cast<uint32_t>(kc2) * 16u + ng2 * 4u);
    a.slot_bytes = round16u(stage1 > stage2 ? stage1 : stage2);
    const size_t budget = kFFNSmemBudget < static_cast<size_t>(dev->max_smem_optin)
                              ? kFFNSmemBudget
                              : static_cast<size_t>(dev->max_smem_optin);
    int nw = 12, ns = 0;
    size_t smem = 0;
    for (; nw >= 8; nw -= 4) {
        for (ns = 4; ns >= 2; --ns) {
            a.off_slots = a.off_bars + round16u(static_cast<uint32_t>(nw * ns) * 8u);
            smem = 128 + static_cast<size_t>(a.off_slots) + static_cast<size_t>(nw) * ns * a.slot_bytes;
            if (smem <= budget) break;
        }
        if (ns >= 2) break;
    }
    if (nw < 8) return cudaSuccess;
    a.ns = ns;
    *unsupported = false;
    cudaError_t err = ensure_dynamic_smem(k, smem);
    if (err != cudaSuccess) return err;
    // cooperative: the CTAs of an expert wait on one another, so the grid
    // starts only when all of them can be resident together
    return launch_coop_pdl(k, dim3(static_cast<unsigned>(a.cpe * n)), dim3(nw * 32), smem, stream, a);
}

}  // namespace smoe
