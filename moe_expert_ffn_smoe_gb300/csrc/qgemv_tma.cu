// Decode GEMV, second design: bulk-copy staging + integer dot products.
//
// Computes the same operations as the S-MoE page "Metal Compute Kernels",
// section "Fused FFN Kernels -- One Simdgroup Per Output Row":
//     hidden[i] = SiLU(gate . x)[i] * (up . x)[i]      (NMAT = 2)
//     out[j]    = (down . hidden)[j]                    (NMAT = 1)
// with w = (code - Z) s / Z and the per-group fold s * (C / Z - Sx).
// One launch covers one expert or several ("Grouped Expert Dispatch"): the
// grid is split into equal slices of CTAs, one slice per expert.
//
// Memory (GB300 layout, not the page's Metal one):
//  * A CTA owns a contiguous range of output rows of one expert and streams
//    it as stages: R consecutive rows of every matrix (one contiguous range
//    per matrix) plus their scales.  Every warp has its own ring of `ns`
//    shared-memory slots which its lane 0 fills with cp.async.bulk copies
//    completing on the slot's mbarrier.  Many threads per SM issue copies:
//    one issuing thread per SM cannot keep HBM busy with copies of a few KB.
//    A warp only ever waits on slots it has filled itself, so the parity of
//    the awaited phase is unambiguous.
//  * The first copies go out before the kernel waits on the previous one
//    (weights are never produced by it), so weight bytes are in flight while
//    x is staged.
//  * x is staged once per CTA, converted to exact integer "digits" (below).
//
// Arithmetic (an exact integer rewrite of the inner dot):
//  * Per 16-byte chunk of codes (32 Q4 or 64 Q2 columns, never more than
//    one group), x is scaled by a power of two 1/q so that its largest
//    magnitude lies in [2^22, 2^23) (one step lower if it would round above
//    XQ_MAX = 8355711) and rounded to an integer xq: |x - xq*q| <= q/2,
//    q <= max|x| / 4177856.
//  * xq is split into three balanced base-256 digits d0 + 256 d1 + 65536 d2,
//    each a signed byte, so sum(code * xq) over a chunk is computed exactly
//    by dp4a (four byte products + add per instruction); codes are
//    separated into bytes with one or two logic ops per 32-bit word (Q4:
//    even nibbles, odd nibbles shifted down; Q2: the four bit pairs), every
//    class on the same grid.
//  * The chunk's dot is taken on the codes minus OFF (8 for Q4, 2 for Q2):
//    C' = sum (code - OFF) xq fits in int32 (|C'| <= 8 * 32 * XQ_MAX), so
//    the modulo-2^32 sums of the digit planes give it exactly.  The chunk
//    adds s * (q/Z * C' + q * Sxq * (OFF - Z)/Z) to the row, which equals
//    s * q * (C/Z - Sxq), the page's fold, with no cancellation between
//    large terms.
// Error: only the rounding of x to xq and the f32 epilogue.  For a chunk
// whose largest |x| = X sits on a weight of magnitude >= s/15 (Q4; s/3 for
// Q2), the rounding error is at most 32 * s * q / 2 <= s X * 3.83e-6 (Q2:
// 64 codes, s X * 7.7e-6), i.e. at most 5.8e-5 (Q2: 2.3e-5) of the
// chunk's sum |w x|; the epilogue adds a few units of 2^-24 of it.
// Non-finite x makes the chunk's q NaN, so the affected outputs are NaN.
#include "qgemv_tma.cuh"

namespace smoe {

// Every warp owns `ns` slots and streams its own stages through them: lane 0
// issues the bulk copies of stage k into slot k % ns, the warp waits on the
// slot's mbarrier, computes the stage's R rows (RPT per team of L lanes)
// and, once all lanes are done with the slot, lane 0 refills it with stage
// k + ns.
template <int BITS, int NMAT, int L, int RPT>
__global__ void __launch_bounds__(512, 1) qgemv_tma(const __grid_constant__ QGArgs a)
{
    using D = DigitFmt<BITS>;
    constexpr int TEAMS = 32 / L;
    constexpr int R = TEAMS * RPT;  // output rows per stage

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
    const int u0 = static_cast<int>(static_cast<long long>(a.units) * bi / a.ctas_per_expert);
    const int u1 = static_cast<int>(static_cast<long long>(a.units) * (bi + 1) / a.ctas_per_expert);
    const int nst = (u1 - u0 + R - 1) / R;
    const int my = warp < nst ? (nst - warp + NW - 1) / NW : 0;  // stages of this warp
    const int KC = a.K / D::CODES_PER_CHUNK;
    const uint32_t row_bytes = static_cast<uint32_t>(KC) * 16u;
    const int ngroups = a.K / a.group;
    const int ns = a.ns;
    const uint32_t bars = sbase + a.off_bars + static_cast<uint32_t>(warp * ns) * 8u;
    const uint32_t slots = sbase + a.off_slots + static_cast<uint32_t>(warp * ns) * a.stage_bytes;
    const uint32_t scales_off = static_cast<uint32_t>(NMAT * R) * row_bytes;

    // this slot's weights (a routed launch resolves them after the wait)
    const uint8_t *mc[2];
    const float *ms[2];
    // lane 0: the bulk copies of this warp's k-th stage into slot k % ns
    auto issue = [&](int k) {
        const int us = u0 + (warp + k * NW) * R;
        const int n = min(R, u1 - us);
        const uint32_t slot = slots + static_cast<uint32_t>(k % ns) * a.stage_bytes;
        const uint32_t bar = bars + static_cast<uint32_t>(k % ns) * 8u;
        const uint32_t cb = static_cast<uint32_t>(n) * row_bytes;
        const uint32_t sb = a.scales_tma ? static_cast<uint32_t>(n * ngroups) * 4u : 0u;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NMAT) * (cb + sb));
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            bulk_g2s(slot + static_cast<uint32_t>(m * R) * row_bytes,
                     mc[m] + static_cast<size_t>(us) * row_bytes, cb, bar);
            if (sb)
                bulk_g2s(slot + scales_off + static_cast<uint32_t>(m * R * ngroups) * 4u,
                         ms[m] + static_cast<size_t>(us) * ngroups, sb, bar);
        }
    };

    // Weights never depend on an earlier kernel: the first stage goes out
    // before waiting for it (unless a routed launch's previous kernel chose
    // them); the rest of the first wave follows the staging of x, whose
    // loads would otherwise queue behind it.
    const int first = my < ns ? my : ns;
    if (!a.route) slot_weights(a, e, NMAT, mc, ms);
    if (lane == 0) {
        for (int i = 0; i < ns; ++i) mbar_init(bars + 8u * i, 1);
        fence_mbar_init();
        if (first > 0 && !a.route) issue(0);
    }
    __syncwarp();

    pdl_wait();
    if (a.route) {
        if (!slot_weights(a, e, NMAT, mc, ms)) {
            fail_route(a, a.y[e], u0, u1);
            return;
        }
        if (lane == 0 && first > 0) issue(0);
        __syncwarp();
    }
    stage_x_digits<BITS>(a.x[e], a.K, a.group, smem, a.off_info);
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (lane == 0)
        for (int k = 1; k < first; ++k) issue(k);
    __syncwarp();

    const int team = lane / L;
    const int u = lane % L;
    const uint32_t info0 = sbase + a.off_info;
    int k = 0;
    bool ok = true;
    for (; k < my; ++k) {
        ok = mbar_wait_bounded(bars + static_cast<uint32_t>(k % ns) * 8u, (k / ns) & 1, a.status, 1u);
        ok = __all_sync(FULL_MASK, ok);
        if (!ok) break;
        const uint32_t slot = slots + static_cast<uint32_t>(k % ns) * a.stage_bytes;
        const int us = u0 + (warp + k * NW) * R;
        const int n = min(R, u1 - us);

        float acc[NMAT][RPT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r) acc[m][r] = 0.f;

        const uint32_t code0 = slot + static_cast<uint32_t>(team) * row_bytes + static_cast<uint32_t>(u) * 16u;
#pragma unroll 2
        for (int c = u; c < KC; c += L) {
            const uint32_t coff = static_cast<uint32_t>(c - u) * 16u;
            const float4 inf = lds128f(info0 + static_cast<uint32_t>(c) * 16u);
            const int g = __float_as_int(inf.z);
            const float qz = inf.x * D::ZINV;
            const uint32_t xc = sbase + static_cast<uint32_t>(c) * D::XSTRIDE;
            uint4 dg[3 * D::NCLASS];
#pragma unroll
            for (int t = 0; t < 3 * D::NCLASS; ++t) dg[t] = lds128u(xc + static_cast<uint32_t>(t) * 16u);
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int ul = r * TEAMS + team;
                    const uint4 cw = lds128u(code0 + static_cast<uint32_t>(m * R + r * TEAMS) * row_bytes + coff);
                    const int C = chunk_dot<BITS>(cw, dg, __float_as_int(inf.w));  // sum (code - OFF) * xq
                    const float sc =
                        a.scales_tma ? lds_f32(slot + scales_off + static_cast<uint32_t>((m * R + ul) * ngroups + g) * 4u)
                                     : ldg_f32(ms[m] + static_cast<size_t>(min(us + ul, u1 - 1)) * ngroups + g);
                    acc[m][r] = fmaf(sc, fmaf(static_cast<float>(C), qz, inf.y), acc[m][r]);
                }
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
                for (int off = L / 2; off > 0; off >>= 1) acc[m][r] += __shfl_xor_sync(FULL_MASK, acc[m][r], off);
        __syncwarp();
        if (lane == 0 && k + ns < my) {
            fence_proxy_async_smem();
            issue(k + ns);
        }
        if (u == 0) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int ul = r * TEAMS + team;
                if (ul < n) {
                    float out = acc[0][r];
                    if (NMAT == 2) out = silu_f32(acc[0][r]) * acc[NMAT - 1][r];
                    a.y[e][us + ul] = out;
                }
            }
        }
    }
    if (!ok && lane == 0) {
        // A copy never completed: wait (bounded) for the ones still in
        // flight before the CTA's shared memory is released.
        const int last = (k + ns < my) ? k + ns : my;
        for (int kk = k; kk < last; ++kk)
            mbar_wait_bounded(bars + static_cast<uint32_t>(kk % ns) * 8u, (kk / ns) & 1, nullptr, 0u);
    }
}

// ---------------------------------------------------------------- host side

namespace {

template <int BITS, int NMAT>
using QGKernel = void (*)(QGArgs);

template <int BITS, int NMAT>
QGKernel<BITS, NMAT> pick_kernel(int L, int rpt)
{
    if (rpt == 2) {
        if (L == 32) return qgemv_tma<BITS, NMAT, 32, 2>;
        if (L == 16) return qgemv_tma<BITS, NMAT, 16, 2>;
        if (L == 8) return qgemv_tma<BITS, NMAT, 8, 2>;
    } else {
        if (L == 32) return qgemv_tma<BITS, NMAT, 32, 1>;
        if (L == 16) return qgemv_tma<BITS, NMAT, 16, 1>;
        if (L == 8) return qgemv_tma<BITS, NMAT, 8, 1>;
    }
    return nullptr;
}

uint32_t round16(uint32_t v) { return (v + 15u) & ~15u; }

constexpr size_t kSmemBudget = 200 * 1024;

// Row-split gate/up kernel: parts per row, used when a CTA would hold fewer
// than kSplitBelow rows (too few stages to keep 12 warps busy).
constexpr int kRowSplit = 2;
constexpr int kSplitBelow = 24;

struct TmaConfig {
    int nw, ns, rpt;
};

// Ring shape for a row range of `max_units` rows: the largest bytes in
// flight that fit the shared-memory budget, preferring 16 warps.
template <int BITS, int NMAT>
bool pick_config(const QGArgs &a, int teams, int max_units, int max_smem, int max_nw, int max_rpt, TmaConfig *out,
                 uint32_t *stage_bytes, uint32_t *off_slots, size_t *smem_out)
{
    using D = DigitFmt<BITS>;
    const int KC = a.K / D::CODES_PER_CHUNK;
    const int ngroups = a.K / a.group;
    const uint32_t row_bytes = static_cast<uint32_t>(KC) * 16u;
    const size_t budget = kSmemBudget < static_cast<size_t>(max_smem) ? kSmemBudget : static_cast<size_t>(max_smem);
    size_t best_flight = 0;
    bool found = false;
    for (int rpt = 1; rpt <= max_rpt; ++rpt) {
        const int R = teams * rpt;
        const int max_stages = (max_units + R - 1) / R;
        const uint32_t sbytes = round16(static_cast<uint32_t>(NMAT * R) * row_bytes +
                                        (a.scales_tma ? static_cast<uint32_t>(NMAT * R * ngroups) * 4u : 0u));
        for (int nw = max_nw; nw >= 8; nw -= 4) {
            const int per_warp = (max_stages + nw - 1) / nw;
            for (int ns = 4; ns >= 1; --ns) {
                if (ns > per_warp && ns > 1) continue;
                const uint32_t offs = a.off_bars + round16(static_cast<uint32_t>(nw * ns) * 8u);
                const size_t smem = 128 + static_cast<size_t>(offs) + static_cast<size_t>(nw) * ns * sbytes;
                if (smem > budget) continue;
                // bytes in flight: all of a warp's stages when its ring holds
                // them, else the slots not being computed on
                const size_t flight = per_warp <= ns ? static_cast<size_t>(nw) * per_warp * sbytes
                                                     : static_cast<size_t>(nw) * (ns - 1) * sbytes;
                if (!found || flight > best_flight) {
                    best_flight = flight;
                    *out = TmaConfig{nw, ns, rpt};
                    *stage_bytes = sbytes;
                    *off_slots = offs;
                    *smem_out = smem;
                    found = true;
                }
                break;  // larger ns for this (rpt, nw) already tried first
            }
        }
    }
    return found;
}

template <int BITS, int NMAT>
cudaError_t launch_tma(QGArgs &a, int n_experts, cudaStream_t stream, bool *unsupported)
{
    using D = DigitFmt<BITS>;
    *unsupported = false;
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const int KC = a.K / D::CODES_PER_CHUNK;
    int L = 0;
    if (KC > 0 && KC % 32 == 0) L = 32;
    else if (KC > 0 && KC % 16 == 0) L = 16;
    else if (KC > 0 && KC % 8 == 0) L = 8;
    if (L == 0 || n_experts < 1 || n_experts > QG_MAX_EXPERTS) {
        *unsupported = true;
        return cudaSuccess;
    }
    const int ngroups = a.K / a.group;
    a.scales_tma = (ngroups % 4 == 0) ? 1 : 0;
    int cpe = dev->sm_count / n_experts;
    if (cpe < 1) cpe = 1;
    a.ctas_per_expert = cpe;
    const int max_units = (a.units + cpe - 1) / cpe;
    a.off_info = static_cast<uint32_t>(KC) * D::XSTRIDE;
    a.off_bars = a.off_info + static_cast<uint32_t>(KC) * 16u;
    TmaConfig cfg;
    size_t smem = 0;
    // Row split (gate/up over few rows per CTA): each lane holds the digits
    // of KC / (32 H) chunks, so 16 warps fit and share H times as many
    // stages; the parts of a row meet in shared memory.
    constexpr int H = kRowSplit;
    if (NMAT == 2 && max_units < kSplitBelow && KC % (32 * H) == 0 && KC / (32 * H) <= 2 &&
        ngroups % (4 * H) == 0) {
        QGArgs av = a;
        av.K = a.K / H;  // the ring carries virtual rows of K / H columns
        const size_t part_bytes = round16(static_cast<uint32_t>(max_units * H * NMAT) * 4u);
        QGKernelFn sk = qgemv_reg_split_kernel(BITS, NMAT, KC / (32 * H), H);
        if (sk && pick_config<BITS, NMAT>(av, 1, max_units * H, dev->max_smem_optin - static_cast<int>(part_bytes),
                                          16, 1, &cfg, &a.stage_bytes, &a.off_slots, &smem)) {
            a.ns = cfg.ns;
            a.off_part = static_cast<uint32_t>(smem - 128);
            smem += part_bytes;
            cudaError_t err = ensure_dynamic_smem(sk, smem);
            if (err != cudaSuccess) return err;
            return launch_pdl(sk, dim3(static_cast<unsigned>(cpe * n_experts)), dim3(cfg.nw * 32), smem, stream, a);
        }
    }
    // Register-digit kernel when a lane's share of the row is at most
    // reg_kernel_max_cpl(BITS) chunks: the largest team (L) that divides KC.
    // One row per team and stage: the 8-expert down projection (4.5 stages
    // per warp with two rows) took 8.1 us, with one row 7.4 us (finer
    // stages even out the warps' last stages).
    int rl = 0;
    for (int l = 32; l >= 8; l >>= 1)
        if (KC % l == 0 && KC / l <= reg_kernel_max_cpl(BITS)) {
            rl = l;
            break;
        }
    if (rl != 0 && a.scales_tma && pick_config<BITS, NMAT>(a, 32 / rl, max_units, dev->max_smem_optin, 12, 1, &cfg,
                                           &a.stage_bytes, &a.off_slots, &smem)) {
        QGKernelFn rk = qgemv_reg_kernel(BITS, NMAT, rl, KC / rl, cfg.rpt);
        if (rk) {
            a.ns = cfg.ns;
            cudaError_t err = ensure_dynamic_smem(rk, smem);
            if (err != cudaSuccess) return err;
            return launch_pdl(rk, dim3(static_cast<unsigned>(cpe * n_experts)), dim3(cfg.nw * 32), smem, stream, a);
        }
    }
    if (!pick_config<BITS, NMAT>(a, 32 / L, max_units, dev->max_smem_optin, 16, 2, &cfg, &a.stage_bytes,
                                 &a.off_slots, &smem)) {
        *unsupported = true;
        return cudaSuccess;
    }
    a.ns = cfg.ns;
    QGKernel<BITS, NMAT> k = pick_kernel<BITS, NMAT>(L, cfg.rpt);
    cudaError_t err = ensure_dynamic_smem(k, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k, dim3(static_cast<unsigned>(cpe * n_experts)), dim3(cfg.nw * 32), smem, stream, a);
}

}  // namespace

namespace {

cudaError_t launch_any(QGArgs &a, int bits, int nmat, int n, cudaStream_t stream, bool *unsupported)
{
    if (bits == 4)
        return nmat == 2 ? launch_tma<4, 2>(a, n, stream, unsupported) : launch_tma<4, 1>(a, n, stream, unsupported);
    return nmat == 2 ? launch_tma<2, 2>(a, n, stream, unsupported) : launch_tma<2, 1>(a, n, stream, unsupported);
}

}  // namespace

cudaError_t launch_qgemv_experts(int bits, int nmat, int n_experts, const uint8_t *const *codes0,
                                 const uint8_t *const *codes1, const float *const *scales0,
                                 const float *const *scales1, const float *const *x, float *const *y,
                                 int units, int K, int group, cudaStream_t stream, bool *unsupported)
{
    QGArgs a = {};
    for (int i = 0; i < n_experts && i < QG_MAX_EXPERTS; ++i) {
        a.codes[0][i] = codes0[i];
        a.codes[1][i] = nmat == 2 ? codes1[i] : codes0[i];
        a.scales[0][i] = scales0[i];
        a.scales[1][i] = nmat == 2 ? scales1[i] : scales0[i];
        a.x[i] = x[i];
        a.y[i] = y[i];
    }
    a.status = device_status_word();
    a.units = units;
    a.K = K;
    a.group = group;
    return launch_any(a, bits, nmat, n_experts, stream, unsupported);
}

cudaError_t launch_qgemv_routed(int bits, int nmat, int n_slots, const uint8_t *const *tab_codes0,
                                const uint8_t *const *tab_codes1, const float *const *tab_scales0,
                                const float *const *tab_scales1, const int *route, int n_route,
                                const float *const *x, float *const *y, int units, int K, int group,
                                cudaStream_t stream, bool *unsupported)
{
    QGArgs a = {};
    for (int i = 0; i < n_slots && i < QG_MAX_EXPERTS; ++i) {
        a.x[i] = x[i];
        a.y[i] = y[i];
    }
    a.route_codes[0] = tab_codes0;
    a.route_codes[1] = nmat == 2 ? tab_codes1 : tab_codes0;
    a.route_scales[0] = tab_scales0;
    a.route_scales[1] = nmat == 2 ? tab_scales1 : tab_scales0;
    a.route = route;
    a.n_route = n_route;
    a.status = device_status_word();
    a.units = units;
    a.K = K;
    a.group = group;
    return launch_any(a, bits, nmat, n_slots, stream, unsupported);
}

}  // namespace smoe
