// The extern "C" entry points declared in include/smoe.h: argument checks
// on the host, then the kernel launches.  Nothing here allocates memory.
#include <mutex>

#include "internal.h"
#include "smoe.h"

namespace smoe {

const DeviceInfo *device_info()
{
    constexpr int kMaxDevices = 64;
    static DeviceInfo cache[kMaxDevices];
    static bool ready[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        DeviceInfo d = {};
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return nullptr;
        cache[dev] = d;
        ready[dev] = true;
    }
    return &cache[dev];
}

}  // namespace smoe

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    const void *p;
    size_t bytes;
};

bool overlap(Span a, Span b)
{
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// True if any output span overlaps any input span or another output span.
bool any_alias(const Span *outs, int nout, const Span *ins, int nin)
{
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlap(outs[i], ins[j])) return true;
        for (int j = i + 1; j < nout; ++j)
            if (overlap(outs[i], outs[j])) return true;
    }
    return false;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? SMOE_OK : SMOE_ERR_LAUNCH; }

// Layout contract of a packed [rows x cols] matrix ("Layout assumptions the
// kernels rely on"): cols % 32 (Q4) / % 64 (Q2), group a positive multiple of
// the same unit dividing cols, cols <= SMOE_MAX_COLS.
int check_q_shape(int bits, int rows, int cols, int group)
{
    if (rows < 0 || cols < 0) return SMOE_ERR_SHAPE;
    if (cols > SMOE_MAX_COLS) return SMOE_ERR_SHAPE;
    const int unit = bits == 4 ? 32 : 64;
    if (cols % unit != 0) return SMOE_ERR_SHAPE;
    if (group <= 0 || group % unit != 0) return SMOE_ERR_SHAPE;
    if (cols > 0 && cols % group != 0) return SMOE_ERR_SHAPE;
    return SMOE_OK;
}

size_t q_bytes(int bits, int rows, int cols)
{
    return static_cast<size_t>(rows) * static_cast<size_t>(cols) * bits / 8;
}

size_t scale_bytes(int rows, int cols, int group)
{
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / group) * sizeof(float);
}

int gate_up_impl(int bits, const uint8_t *gc, const float *gs, const uint8_t *uc, const float *us,
                 const float *x, float *hidden, int d_ff, int d_model, int group, void *stream)
{
    int st = check_q_shape(bits, d_ff, d_model, group);
    if (st != SMOE_OK) return st;
    if (d_ff == 0) return SMOE_OK;
    if (!hidden) return SMOE_ERR_NULL;
    if (!aligned16(hidden)) return SMOE_ERR_ALIGN;
    if (d_model > 0) {
        if (!gc || !gs || !uc || !us || !x) return SMOE_ERR_NULL;
        if (!aligned16(gc) || !aligned16(uc) || !aligned16(gs) || !aligned16(us) || !aligned16(x))
            return SMOE_ERR_ALIGN;
    }
    const Span out[1] = {{hidden, static_cast<size_t>(d_ff) * sizeof(float)}};
    const Span in[5] = {{gc, q_bytes(bits, d_ff, d_model)},
                        {gs, scale_bytes(d_ff, d_model, group)},
                        {uc, q_bytes(bits, d_ff, d_model)},
                        {us, scale_bytes(d_ff, d_model, group)},
                        {x, static_cast<size_t>(d_model) * sizeof(float)}};
    if (any_alias(out, 1, in, 5)) return SMOE_ERR_ALIAS;
    const uint8_t *codes[2] = {gc, uc};
    const float *scales[2] = {gs, us};
    return to_status(smoe::launch_qgemv(bits, 2, codes, scales, x, hidden, d_ff, d_model, group,
                                        static_cast<cudaStream_t>(stream)));
}

int down_impl(int bits, const uint8_t *dc, const float *ds, const float *hidden, float *out,
              int d_model, int d_ff, int group, void *stream)
{
    int st = check_q_shape(bits, d_model, d_ff, group);
    if (st != SMOE_OK) return st;
    if (d_model == 0) return SMOE_OK;
    if (!out) return SMOE_ERR_NULL;
    if (!aligned16(out)) return SMOE_ERR_ALIGN;
    if (d_ff > 0) {
        if (!dc || !ds || !hidden) return SMOE_ERR_NULL;
        if (!aligned16(dc) || !aligned16(ds) || !aligned16(hidden)) return SMOE_ERR_ALIGN;
    }
    const Span o[1] = {{out, static_cast<size_t>(d_model) * sizeof(float)}};
    const Span in[3] = {{dc, q_bytes(bits, d_model, d_ff)},
                        {ds, scale_bytes(d_model, d_ff, group)},
                        {hidden, static_cast<size_t>(d_ff) * sizeof(float)}};
    if (any_alias(o, 1, in, 3)) return SMOE_ERR_ALIAS;
    const uint8_t *codes[2] = {dc, dc};
    const float *scales[2] = {ds, ds};
    return to_status(smoe::launch_qgemv(bits, 1, codes, scales, hidden, out, d_model, d_ff, group,
                                        static_cast<cudaStream_t>(stream)));
}

constexpr int kExpertsPerLaunch = 64;

int launch_grouped(int bits, int nmat, int n, const uint8_t *const *c0, const float *const *s0,
                   const uint8_t *const *c1, const float *const *s1, const float *x, float *y, int units, int K,
                   int group, cudaStream_t s);

// Grouped calls: per-expert checks, then launches of up to 64 experts each
// (experts of one launch share the grid; a shape the grouped kernel does not
// take is run expert by expert with the single-expert launcher).
int experts_impl(int bits, int nmat, int n, const uint8_t *const *c0, const float *const *s0,
                 const uint8_t *const *c1, const float *const *s1, const float *x, float *y, int units, int K,
                 int group, void *stream)
{
    if (n < 0) return SMOE_ERR_SHAPE;
    int st = check_q_shape(bits, units, K, group);
    if (st != SMOE_OK) return st;
    if (n == 0 || units == 0) return SMOE_OK;
    if (!c0 || !s0 || (nmat == 2 && (!c1 || !s1))) return SMOE_ERR_NULL;
    if (!y) return SMOE_ERR_NULL;
    if (!aligned16(y)) return SMOE_ERR_ALIGN;
    // x: one shared vector for gate/up, one row per expert for down
    const size_t x_bytes = static_cast<size_t>(K) * sizeof(float) * (nmat == 2 ? 1 : static_cast<size_t>(n));
    const Span out = {y, static_cast<size_t>(n) * static_cast<size_t>(units) * sizeof(float)};
    if (K > 0) {
        if (!x) return SMOE_ERR_NULL;
        if (!aligned16(x)) return SMOE_ERR_ALIGN;
        if (overlap(out, Span{x, x_bytes})) return SMOE_ERR_ALIAS;
        for (int e = 0; e < n; ++e) {
            const uint8_t *cs[2] = {c0[e], nmat == 2 ? c1[e] : c0[e]};
            const float *ss[2] = {s0[e], nmat == 2 ? s1[e] : s0[e]};
            for (int m = 0; m < nmat; ++m) {
                if (!cs[m] || !ss[m]) return SMOE_ERR_NULL;
                if (!aligned16(cs[m]) || !aligned16(ss[m])) return SMOE_ERR_ALIGN;
                if (overlap(out, Span{cs[m], q_bytes(bits, units, K)}) ||
                    overlap(out, Span{ss[m], scale_bytes(units, K, group)}))
                    return SMOE_ERR_ALIAS;
            }
        }
    }
    return launch_grouped(bits, nmat, n, c0, s0, c1, s1, x, y, units, K, group, static_cast<cudaStream_t>(stream));
}

// The launches of a grouped call whose arguments have been checked.
int launch_grouped(int bits, int nmat, int n, const uint8_t *const *c0, const float *const *s0,
                   const uint8_t *const *c1, const float *const *s1, const float *x, float *y, int units, int K,
                   int group, cudaStream_t s)
{
    if (n == 0 || units == 0) return SMOE_OK;
    const float *xs[kExpertsPerLaunch];
    float *ys[kExpertsPerLaunch];
    for (int e0 = 0; e0 < n; e0 += kExpertsPerLaunch) {
        const int cnt = (n - e0) < kExpertsPerLaunch ? (n - e0) : kExpertsPerLaunch;
        for (int i = 0; i < cnt; ++i) {
            xs[i] = nmat == 2 ? x : (x ? x + static_cast<size_t>(e0 + i) * K : nullptr);
            ys[i] = y + static_cast<size_t>(e0 + i) * units;
        }
        bool unsupported = true;
        cudaError_t err = cudaSuccess;
        if (K > 0)
            err = smoe::launch_qgemv_experts(bits, nmat, cnt, c0 + e0, nmat == 2 ? c1 + e0 : c0 + e0, s0 + e0,
                                             nmat == 2 ? s1 + e0 : s0 + e0, xs, ys, units, K, group, s,
                                             &unsupported);
        if (err != cudaSuccess) return SMOE_ERR_LAUNCH;
        if (unsupported) {
            for (int i = 0; i < cnt; ++i) {
                const uint8_t *codes[2] = {c0[e0 + i], nmat == 2 ? c1[e0 + i] : c0[e0 + i]};
                const float *scales[2] = {s0[e0 + i], nmat == 2 ? s1[e0 + i] : s0[e0 + i]};
                err = smoe::launch_qgemv(bits, nmat, codes, scales, xs[i], ys[i], units, K, group, s);
                if (err != cudaSuccess) return SMOE_ERR_LAUNCH;
            }
        }
    }
    return SMOE_OK;
}

size_t ffn_workspace_bytes(int n, int d_ff)
{
    if (d_ff < 0) return static_cast<size_t>(-1);
    if (n <= 0) return 0;
    const size_t e = static_cast<size_t>(n < kExpertsPerLaunch ? n : kExpertsPerLaunch);
    const size_t b = SMOE_FFN_SYNC_BYTES + e * static_cast<size_t>(d_ff) * sizeof(float);
    return (b + 255u) & ~static_cast<size_t>(255u);
}

// smoe_experts_ffn_q4/q2: checks, then per 64 experts the one-launch
// kernel, or gate/up into the workspace followed by down.
int experts_ffn_impl(int bits, int n, const uint8_t *const *gc, const float *const *gs, const uint8_t *const *uc,
                     const float *const *us, const uint8_t *const *dc, const float *const *ds, const float *x,
                     float *out, int d_model, int d_ff, int group, void *workspace, size_t ws_bytes, void *stream)
{
    if (n < 0) return SMOE_ERR_SHAPE;
    int st = check_q_shape(bits, d_ff, d_model, group);
    if (st != SMOE_OK) return st;
    st = check_q_shape(bits, d_model, d_ff, group);
    if (st != SMOE_OK) return st;
    if (n == 0 || d_model == 0) return SMOE_OK;
    if (!gc || !gs || !uc || !us || !dc || !ds || !x || !out) return SMOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(out)) return SMOE_ERR_ALIGN;
    const size_t need = ffn_workspace_bytes(n, d_ff);
    if (!workspace || ws_bytes < need) return SMOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SMOE_ERR_ALIGN;
    const Span o = {out, static_cast<size_t>(n) * static_cast<size_t>(d_model) * sizeof(float)};
    const Span w = {workspace, need};
    const Span xi = {x, static_cast<size_t>(d_model) * sizeof(float)};
    if (overlap(o, xi) || overlap(o, w) || overlap(w, xi)) return SMOE_ERR_ALIAS;
    for (int e = 0; e < n; ++e) {
        const void *ptrs[6] = {gc[e], gs[e], uc[e], us[e], dc[e], ds[e]};
        for (const void *p : ptrs) {
            if (!p) return SMOE_ERR_NULL;
            if (!aligned16(p)) return SMOE_ERR_ALIGN;
        }
        const Span ins[6] = {{gc[e], q_bytes(bits, d_ff, d_model)}, {gs[e], scale_bytes(d_ff, d_model, group)},
                             {uc[e], q_bytes(bits, d_ff, d_model)}, {us[e], scale_bytes(d_ff, d_model, group)},
                             {dc[e], q_bytes(bits, d_model, d_ff)}, {ds[e], scale_bytes(d_model, d_ff, group)}};
        for (const Span &in : ins)
            if (overlap(o, in) || overlap(w, in)) return SMOE_ERR_ALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned *sync = static_cast<unsigned *>(workspace);
    float *hidden = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + SMOE_FFN_SYNC_BYTES);
    for (int e0 = 0; e0 < n; e0 += kExpertsPerLaunch) {
        const int cnt = (n - e0) < kExpertsPerLaunch ? (n - e0) : kExpertsPerLaunch;
        float *o0 = out + static_cast<size_t>(e0) * d_model;
        bool unsupported = true;
        cudaError_t err = cudaSuccess;
        if (d_ff > 0)
            err = smoe::launch_expert_ffn(bits, cnt, gc + e0, gs + e0, uc + e0, us + e0, dc + e0, ds + e0, x,
                                          hidden, o0, sync, d_model, d_ff, group, s, &unsupported);
        if (err != cudaSuccess) return SMOE_ERR_LAUNCH;
        if (unsupported) {
            st = launch_grouped(bits, 2, cnt, gc + e0, gs + e0, uc + e0, us + e0, x, hidden, d_ff, d_model, group,
                                s);
            if (st != SMOE_OK) return st;
            st = launch_grouped(bits, 1, cnt, dc + e0, ds + e0, nullptr, nullptr, hidden, o0, d_model, d_ff, group,
                                s);
            if (st != SMOE_OK) return st;
        }
    }
    return SMOE_OK;
}

// ffn_batch_q4/q2: checks, then the token-batch launches.
int ffn_batch_impl(int bits, const uint8_t *gate_codes, const float *gate_scales, const uint8_t *up_codes,
                 const float *up_scales, const uint8_t *down_codes, const float *down_scales,
                 const float *X, float *Y, int T, int d_model, int d_ff, int group,
                 void *workspace, size_t workspace_bytes, void *stream)
{
    if (T < 0) return SMOE_ERR_SHAPE;
    int st = check_q_shape(bits, d_ff, d_model, group);
    if (st != SMOE_OK) return st;
    st = check_q_shape(bits, d_model, d_ff, group);
    if (st != SMOE_OK) return st;
    if (T == 0 || d_model == 0) return SMOE_OK;
    if (!X || !Y) return SMOE_ERR_NULL;
    if (!aligned16(X) || !aligned16(Y)) return SMOE_ERR_ALIGN;
    if (d_ff > 0) {
        if (!gate_codes || !gate_scales || !up_codes || !up_scales || !down_codes || !down_scales)
            return SMOE_ERR_NULL;
        if (!aligned16(gate_codes) || !aligned16(gate_scales) || !aligned16(up_codes) ||
            !aligned16(up_scales) || !aligned16(down_codes) || !aligned16(down_scales))
            return SMOE_ERR_ALIGN;
    }
    const size_t need = smoe::ffn_batch_workspace(T, d_model, d_ff, group);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return SMOE_ERR_WORKSPACE;
        if (!aligned16(workspace)) return SMOE_ERR_ALIGN;
    }
    const size_t xy = static_cast<size_t>(T) * static_cast<size_t>(d_model) * sizeof(float);
    const Span outs[2] = {{Y, xy}, {workspace, need}};
    const Span ins[7] = {{gate_codes, q_bytes(bits, d_ff, d_model)},
                         {gate_scales, scale_bytes(d_ff, d_model, group)},
                         {up_codes, q_bytes(bits, d_ff, d_model)},
                         {up_scales, scale_bytes(d_ff, d_model, group)},
                         {down_codes, q_bytes(bits, d_model, d_ff)},
                         {down_scales, scale_bytes(d_model, d_ff, group)},
                         {X, xy}};
    if (any_alias(outs, 2, ins, 7)) return SMOE_ERR_ALIAS;
    const uint8_t *gu_codes[2] = {gate_codes, up_codes};
    const float *gu_scales[2] = {gate_scales, up_scales};
    return to_status(smoe::launch_ffn_batch(bits, gu_codes, gu_scales, down_codes, down_scales, X, Y, T,
                                            d_model, d_ff, group, workspace,
                                            static_cast<cudaStream_t>(stream)));
}

// smoe_experts_ffn_batch_q4/q2: per-expert checks, then the grouped
// token-batch launches.
int experts_batch_impl(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                       const uint8_t *const *uc, const float *const *us, const uint8_t *const *dc,
                       const float *const *ds, const float *const *X, float *const *Y, const int *T, int d_model,
                       int d_ff, int group, void *workspace, size_t ws_bytes, void *stream)
{
    if (n < 0) return SMOE_ERR_SHAPE;
    int st = check_q_shape(bits, d_ff, d_model, group);
    if (st != SMOE_OK) return st;
    st = check_q_shape(bits, d_model, d_ff, group);
    if (st != SMOE_OK) return st;
    if (n == 0 || d_model == 0) return SMOE_OK;
    if (!T) return SMOE_ERR_NULL;
    bool any = false;
    for (int e = 0; e < n; ++e) {
        if (T[e] < 0) return SMOE_ERR_SHAPE;
        any = any || T[e] > 0;
    }
    if (!any) return SMOE_OK;
    if (!gc || !gs || !uc || !us || !dc || !ds || !X || !Y) return SMOE_ERR_NULL;
    const size_t need = smoe::ffn_batch_workspace_experts(n, T, d_model, d_ff, group);
    if (need > 0) {
        if (!workspace || ws_bytes < need) return SMOE_ERR_WORKSPACE;
        if (!aligned16(workspace)) return SMOE_ERR_ALIGN;
    }
    const Span w = {workspace, need};
    for (int e = 0; e < n; ++e) {
        if (T[e] == 0) continue;
        const void *ptrs[8] = {gc[e], gs[e], uc[e], us[e], dc[e], ds[e], X[e], Y[e]};
        for (const void *p : ptrs) {
            if (!p) return SMOE_ERR_NULL;
            if (!aligned16(p)) return SMOE_ERR_ALIGN;
        }
    }
    // every output against every input, the workspace and the other outputs
    for (int e = 0; e < n; ++e) {
        if (T[e] == 0) continue;
        const Span o = {Y[e], static_cast<size_t>(T[e]) * static_cast<size_t>(d_model) * sizeof(float)};
        if (need > 0 && overlap(o, w)) return SMOE_ERR_ALIAS;
        for (int f = 0; f < n; ++f) {
            if (T[f] == 0) continue;
            const Span ins[7] = {{gc[f], q_bytes(bits, d_ff, d_model)}, {gs[f], scale_bytes(d_ff, d_model, group)},
                                 {uc[f], q_bytes(bits, d_ff, d_model)}, {us[f], scale_bytes(d_ff, d_model, group)},
                                 {dc[f], q_bytes(bits, d_model, d_ff)}, {ds[f], scale_bytes(d_model, d_ff, group)},
                                 {X[f], static_cast<size_t>(T[f]) * static_cast<size_t>(d_model) * sizeof(float)}};
            for (const Span &in : ins)
                if (overlap(o, in) || (need > 0 && overlap(w, in))) return SMOE_ERR_ALIAS;
            if (f > e && overlap(o, Span{Y[f], static_cast<size_t>(T[f]) * static_cast<size_t>(d_model) *
                                                   sizeof(float)}))
                return SMOE_ERR_ALIAS;
        }
    }
    return to_status(smoe::launch_ffn_batch_experts(bits, n, gc, gs, uc, us, dc, ds, X, Y, T, d_model, d_ff, group,
                                                    workspace, static_cast<cudaStream_t>(stream)));
}

// Routed FFN: hidden[k x d_ff] in the workspace, out[k x d_model].
size_t routed_hidden_bytes(int k, int d_ff)
{
    const size_t b = static_cast<size_t>(k) * static_cast<size_t>(d_ff) * sizeof(float);
    return (b + 255u) & ~static_cast<size_t>(255u);
}

int experts_ffn_routed_impl(int bits, int n_experts, int k, const uint8_t *const *gc, const float *const *gs,
                            const uint8_t *const *uc, const float *const *us, const uint8_t *const *dc,
                            const float *const *ds, const int *top_idx, const float *x, float *out, int d_model,
                            int d_ff, int group, void *workspace, size_t workspace_bytes, void *stream)
{
    if (n_experts < 0 || k < 0 || k > SMOE_MAX_ROUTED_SLOTS) return SMOE_ERR_SHAPE;
    int st = check_q_shape(bits, d_ff, d_model, group);
    if (st != SMOE_OK) return st;
    st = check_q_shape(bits, d_model, d_ff, group);
    if (st != SMOE_OK) return st;
    // rows the bulk-copy decode kernels take: whole multiples of 8 chunks of
    // 16 bytes, at most 8192 columns (their staging then always fits)
    const int unit = bits == 4 ? 256 : 512;
    if (d_model % unit || d_ff % unit || d_model > 8192 || d_ff > 8192) return SMOE_ERR_SHAPE;
    if (k == 0 || d_model == 0) return SMOE_OK;
    if (n_experts == 0) return SMOE_ERR_SHAPE;  // no index could be valid
    if (!out || !top_idx) return SMOE_ERR_NULL;
    if (!aligned16(out) || (reinterpret_cast<uintptr_t>(top_idx) & 3u)) return SMOE_ERR_ALIGN;
    const size_t out_bytes = static_cast<size_t>(k) * static_cast<size_t>(d_model) * sizeof(float);
    const Span idx_span = {top_idx, static_cast<size_t>(k) * sizeof(int)};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d_ff == 0) {
        // every output is an empty sum
        if (overlap(Span{out, out_bytes}, idx_span)) return SMOE_ERR_ALIAS;
        return to_status(cudaMemsetAsync(out, 0, out_bytes, s));
    }
    if (!gc || !gs || !uc || !us || !dc || !ds || !x) return SMOE_ERR_NULL;
    const void *tabs[6] = {gc, gs, uc, us, dc, ds};
    for (const void *t : tabs)
        if (reinterpret_cast<uintptr_t>(t) & 7u) return SMOE_ERR_ALIGN;
    if (!aligned16(x)) return SMOE_ERR_ALIGN;
    const size_t need = routed_hidden_bytes(k, d_ff);
    if (!workspace || workspace_bytes < need) return SMOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SMOE_ERR_ALIGN;
    const size_t tab_bytes = static_cast<size_t>(n_experts) * sizeof(void *);
    const Span outs[2] = {{out, out_bytes}, {workspace, need}};
    const Span ins[8] = {{x, static_cast<size_t>(d_model) * sizeof(float)}, idx_span,
                         {gc, tab_bytes}, {gs, tab_bytes}, {uc, tab_bytes}, {us, tab_bytes},
                         {dc, tab_bytes}, {ds, tab_bytes}};
    if (any_alias(outs, 2, ins, 8)) return SMOE_ERR_ALIAS;
    float *hidden = static_cast<float *>(workspace);
    const float *xs[SMOE_MAX_ROUTED_SLOTS];
    float *ys[SMOE_MAX_ROUTED_SLOTS];
    for (int e = 0; e < k; ++e) {
        xs[e] = x;
        ys[e] = hidden + static_cast<size_t>(e) * d_ff;
    }
    bool unsupported = true;
    cudaError_t err = smoe::launch_qgemv_routed(bits, 2, k, gc, uc, gs, us, top_idx, n_experts, xs, ys, d_ff,
                                                d_model, group, s, &unsupported);
    if (unsupported) return SMOE_ERR_SHAPE;
    if (err != cudaSuccess) return SMOE_ERR_LAUNCH;
    for (int e = 0; e < k; ++e) {
        xs[e] = hidden + static_cast<size_t>(e) * d_ff;
        ys[e] = out + static_cast<size_t>(e) * d_model;
    }
    err = smoe::launch_qgemv_routed(bits, 1, k, dc, dc, ds, ds, top_idx, n_experts, xs, ys, d_model, d_ff, group,
                                    s, &unsupported);
    if (unsupported) return SMOE_ERR_SHAPE;
    return to_status(err);
}

}  // namespace

extern "C" {

size_t smoe_experts_ffn_workspace_bytes(int n_experts, int d_ff) { return ffn_workspace_bytes(n_experts, d_ff); }

int smoe_experts_ffn_q4(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                        const uint8_t *const *up_codes, const float *const *up_scales,
                        const uint8_t *const *down_codes, const float *const *down_scales, const float *x,
                        float *out, int d_model, int d_ff, int group, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return experts_ffn_impl(4, n_experts, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
                            x, out, d_model, d_ff, group, workspace, workspace_bytes, stream);
}

int smoe_experts_ffn_q2(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                        const uint8_t *const *up_codes, const float *const *up_scales,
                        const uint8_t *const *down_codes, const float *const *down_scales, const float *x,
                        float *out, int d_model, int d_ff, int group, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return experts_ffn_impl(2, n_experts, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
                            x, out, d_model, d_ff, group, workspace, workspace_bytes, stream);
}

int smoe_experts_gate_up_q4(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                            const uint8_t *const *up_codes, const float *const *up_scales, const float *x,
                            float *hidden, int d_ff, int d_model, int group, void *stream)
{
    return experts_impl(4, 2, n_experts, gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff,
                        d_model, group, stream);
}

int smoe_experts_gate_up_q2(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                            const uint8_t *const *up_codes, const float *const *up_scales, const float *x,
                            float *hidden, int d_ff, int d_model, int group, void *stream)
{
    return experts_impl(2, 2, n_experts, gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff,
                        d_model, group, stream);
}

int smoe_experts_down_q4(int n_experts, const uint8_t *const *down_codes, const float *const *down_scales,
                         const float *hidden, float *out, int d_model, int d_ff, int group, void *stream)
{
    return experts_impl(4, 1, n_experts, down_codes, down_scales, nullptr, nullptr, hidden, out, d_model,
                        d_ff, group, stream);
}

int smoe_experts_down_q2(int n_experts, const uint8_t *const *down_codes, const float *const *down_scales,
                         const float *hidden, float *out, int d_model, int d_ff, int group, void *stream)
{
    return experts_impl(2, 1, n_experts, down_codes, down_scales, nullptr, nullptr, hidden, out, d_model,
                        d_ff, group, stream);
}

int smoe_abi_version(void) { return SMOE_ABI_VERSION; }

const char *smoe_status_string(int status)
{
    switch (status) {
    case SMOE_OK: return "ok";
    case SMOE_ERR_NULL: return "a required pointer is NULL";
    case SMOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case SMOE_ERR_SHAPE: return "sizes break the layout contract or the limits";
    case SMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case SMOE_ERR_LAUNCH: return "CUDA launch or device query failed";
    case SMOE_ERR_TIMEOUT: return "a device-side bounded wait gave up";
    case SMOE_ERR_ALIAS: return "an output overlaps an input or another output";
    case SMOE_ERR_MEMORY: return "a buffer is not accessible from the device";
    case SMOE_ERR_ROUTE: return "a device-side expert index or table entry was invalid";
    default: return "unknown status";
    }
}

int smoe_gate_up_q4(const uint8_t *gate_codes, const float *gate_scales, const uint8_t *up_codes,
                    const float *up_scales, const float *x, float *hidden, int d_ff, int d_model,
                    int group, void *stream)
{
    return gate_up_impl(4, gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model,
                        group, stream);
}

int smoe_gate_up_q2(const uint8_t *gate_codes, const float *gate_scales, const uint8_t *up_codes,
                    const float *up_scales, const float *x, float *hidden, int d_ff, int d_model,
                    int group, void *stream)
{
    return gate_up_impl(2, gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model,
                        group, stream);
}

int smoe_down_q4(const uint8_t *down_codes, const float *down_scales, const float *hidden,
                 float *out, int d_model, int d_ff, int group, void *stream)
{
    return down_impl(4, down_codes, down_scales, hidden, out, d_model, d_ff, group, stream);
}

int smoe_down_q2(const uint8_t *down_codes, const float *down_scales, const float *hidden,
                 float *out, int d_model, int d_ff, int group, void *stream)
{
    return down_impl(2, down_codes, down_scales, hidden, out, d_model, d_ff, group, stream);
}

int matvec_bf16(const uint16_t *w, const float *x, float *y, int rows, int cols, void *stream)
{
    if (rows < 0 || cols < 0 || cols > SMOE_MAX_COLS || cols % 8 != 0) return SMOE_ERR_SHAPE;
    if (rows == 0) return SMOE_OK;
    if (!y) return SMOE_ERR_NULL;
    if (!aligned16(y)) return SMOE_ERR_ALIGN;
    if (cols > 0) {
        if (!w || !x) return SMOE_ERR_NULL;
        if (!aligned16(w) || !aligned16(x)) return SMOE_ERR_ALIGN;
    }
    const Span o[1] = {{y, static_cast<size_t>(rows) * sizeof(float)}};
    const Span in[2] = {{w, static_cast<size_t>(rows) * static_cast<size_t>(cols) * 2},
                        {x, static_cast<size_t>(cols) * sizeof(float)}};
    if (any_alias(o, 1, in, 2)) return SMOE_ERR_ALIAS;
    return to_status(smoe::launch_bf16_gemv(w, x, y, rows, cols, static_cast<cudaStream_t>(stream)));
}

int matvec_bf16_batch(int n, const uint16_t *const *w, const float *const *x, float *const *y,
                      const int *rows, const int *cols, void *stream)
{
    if (n < 0) return SMOE_ERR_SHAPE;
    if (n == 0) return SMOE_OK;
    if (!w || !x || !y || !rows || !cols) return SMOE_ERR_NULL;
    for (int i = 0; i < n; ++i) {
        if (rows[i] < 0 || cols[i] < 0 || cols[i] > SMOE_MAX_COLS || cols[i] % 8 != 0) return SMOE_ERR_SHAPE;
        if (rows[i] == 0) continue;
        if (!y[i]) return SMOE_ERR_NULL;
        if (!aligned16(y[i])) return SMOE_ERR_ALIGN;
        if (cols[i] > 0) {
            if (!w[i] || !x[i]) return SMOE_ERR_NULL;
            if (!aligned16(w[i]) || !aligned16(x[i])) return SMOE_ERR_ALIGN;
        }
    }
    // every output against every input and every other output
    for (int i = 0; i < n; ++i) {
        if (rows[i] == 0) continue;
        const Span o = {y[i], static_cast<size_t>(rows[i]) * sizeof(float)};
        for (int j = 0; j < n; ++j) {
            if (rows[j] == 0) continue;
            if (j > i && overlap(o, Span{y[j], static_cast<size_t>(rows[j]) * sizeof(float)})) return SMOE_ERR_ALIAS;
            if (cols[j] == 0) continue;
            if (overlap(o, Span{w[j], static_cast<size_t>(rows[j]) * static_cast<size_t>(cols[j]) * 2}) ||
                overlap(o, Span{x[j], static_cast<size_t>(cols[j]) * sizeof(float)}))
                return SMOE_ERR_ALIAS;
        }
    }
    return to_status(smoe::launch_bf16_gemv_batch(n, w, x, y, rows, cols, static_cast<cudaStream_t>(stream)));
}

size_t smoe_ffn_batch_workspace_bytes(int T, int d_model, int d_ff, int group)
{
    if (check_q_shape(4, d_ff, d_model, group) != SMOE_OK ||
        check_q_shape(4, d_model, d_ff, group) != SMOE_OK)
        return static_cast<size_t>(-1);
    if (T <= 0) return 0;
    return smoe::ffn_batch_workspace(T, d_model, d_ff, group);
}

int ffn_batch_q4(const uint8_t *gate_codes, const float *gate_scales, const uint8_t *up_codes,
                 const float *up_scales, const uint8_t *down_codes, const float *down_scales,
                 const float *X, float *Y, int T, int d_model, int d_ff, int group,
                 void *workspace, size_t workspace_bytes, void *stream)
{
    return ffn_batch_impl(4, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                          d_model, d_ff, group, workspace, workspace_bytes, stream);
}

int ffn_batch_q2(const uint8_t *gate_codes, const float *gate_scales, const uint8_t *up_codes,
                 const float *up_scales, const uint8_t *down_codes, const float *down_scales,
                 const float *X, float *Y, int T, int d_model, int d_ff, int group,
                 void *workspace, size_t workspace_bytes, void *stream)
{
    return ffn_batch_impl(2, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                          d_model, d_ff, group, workspace, workspace_bytes, stream);
}

size_t smoe_experts_ffn_batch_workspace_bytes(int n_experts, const int *T, int d_model, int d_ff, int group)
{
    if (n_experts <= 0) return 0;
    if (!T) return static_cast<size_t>(-1);
    // the Q4 layout rules (Q2's are stricter: a Q2 shape passes them too)
    if (check_q_shape(4, d_ff, d_model, group) != SMOE_OK || check_q_shape(4, d_model, d_ff, group) != SMOE_OK)
        return static_cast<size_t>(-1);
    for (int e = 0; e < n_experts; ++e)
        if (T[e] < 0) return static_cast<size_t>(-1);
    return smoe::ffn_batch_workspace_experts(n_experts, T, d_model, d_ff, group);
}

int smoe_experts_ffn_batch_q4(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                              const uint8_t *const *up_codes, const float *const *up_scales,
                              const uint8_t *const *down_codes, const float *const *down_scales,
                              const float *const *X, float *const *Y, const int *T, int d_model, int d_ff,
                              int group, void *workspace, size_t workspace_bytes, void *stream)
{
    return experts_batch_impl(4, n_experts, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
                              X, Y, T, d_model, d_ff, group, workspace, workspace_bytes, stream);
}

int smoe_experts_ffn_batch_q2(int n_experts, const uint8_t *const *gate_codes, const float *const *gate_scales,
                              const uint8_t *const *up_codes, const float *const *up_scales,
                              const uint8_t *const *down_codes, const float *const *down_scales,
                              const float *const *X, float *const *Y, const int *T, int d_model, int d_ff,
                              int group, void *workspace, size_t workspace_bytes, void *stream)
{
    return experts_batch_impl(2, n_experts, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
                              X, Y, T, d_model, d_ff, group, workspace, workspace_bytes, stream);
}

size_t smoe_experts_ffn_routed_workspace_bytes(int k, int d_ff)
{
    if (k < 0 || k > SMOE_MAX_ROUTED_SLOTS || d_ff < 0) return static_cast<size_t>(-1);
    return routed_hidden_bytes(k, d_ff);
}

int smoe_experts_ffn_routed_q4(int n_experts, int k, const uint8_t *const *gate_codes,
                               const float *const *gate_scales, const uint8_t *const *up_codes,
                               const float *const *up_scales, const uint8_t *const *down_codes,
                               const float *const *down_scales, const int *top_idx, const float *x, float *out,
                               int d_model, int d_ff, int group, void *workspace, size_t workspace_bytes,
                               void *stream)
{
    return experts_ffn_routed_impl(4, n_experts, k, gate_codes, gate_scales, up_codes, up_scales, down_codes,
                                   down_scales, top_idx, x, out, d_model, d_ff, group, workspace, workspace_bytes,
                                   stream);
}

int smoe_experts_ffn_routed_q2(int n_experts, int k, const uint8_t *const *gate_codes,
                               const float *const *gate_scales, const uint8_t *const *up_codes,
                               const float *const *up_scales, const uint8_t *const *down_codes,
                               const float *const *down_scales, const int *top_idx, const float *x, float *out,
                               int d_model, int d_ff, int group, void *workspace, size_t workspace_bytes,
                               void *stream)
{
    return experts_ffn_routed_impl(2, n_experts, k, gate_codes, gate_scales, up_codes, up_scales, down_codes,
                                   down_scales, top_idx, x, out, d_model, d_ff, group, workspace, workspace_bytes,
                                   stream);
}

int smoe_route_topk_bf16(const uint16_t *gate_w, const float *x, int n_experts, int d_model, int k, float *logits,
                         int *top_idx, float *top_w, void *stream)
{
    if (n_experts < 1 || n_experts > SMOE_MAX_ROUTE_EXPERTS) return SMOE_ERR_SHAPE;
    if (k < 1 || k > n_experts || k > SMOE_MAX_TOP_K) return SMOE_ERR_SHAPE;
    if (d_model < 0 || d_model > SMOE_MAX_COLS || d_model % 8 != 0) return SMOE_ERR_SHAPE;
    if (!logits || !top_idx || !top_w) return SMOE_ERR_NULL;
    if (d_model > 0 && (!gate_w || !x)) return SMOE_ERR_NULL;
    if (!aligned16(logits) || (d_model > 0 && (!aligned16(gate_w) || !aligned16(x)))) return SMOE_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(top_idx) & 3u) || (reinterpret_cast<uintptr_t>(top_w) & 3u))
        return SMOE_ERR_ALIGN;
    const Span outs[3] = {{logits, static_cast<size_t>(n_experts) * sizeof(float)},
                          {top_idx, static_cast<size_t>(k) * sizeof(int)},
                          {top_w, static_cast<size_t>(k) * sizeof(float)}};
    const Span ins[2] = {{gate_w, static_cast<size_t>(n_experts) * static_cast<size_t>(d_model) * 2},
                         {x, static_cast<size_t>(d_model) * sizeof(float)}};
    if (any_alias(outs, 3, ins, d_model > 0 ? 2 : 0)) return SMOE_ERR_ALIAS;
    return to_status(smoe::launch_route(gate_w, x, n_experts, d_model, k, logits, top_idx, top_w,
                                        static_cast<cudaStream_t>(stream)));
}

int smoe_combine(int k, const float *expert_out, const float *top_w, float *out, int d_model, void *stream)
{
    if (k < 0 || d_model < 0) return SMOE_ERR_SHAPE;
    if (d_model == 0) return SMOE_OK;
    if (!out || (k > 0 && (!expert_out || !top_w))) return SMOE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) || (k > 0 && ((reinterpret_cast<uintptr_t>(expert_out) & 3u) ||
                                                             (reinterpret_cast<uintptr_t>(top_w) & 3u))))
        return SMOE_ERR_ALIGN;
    const Span o[1] = {{out, static_cast<size_t>(d_model) * sizeof(float)}};
    const Span ins[2] = {{expert_out, static_cast<size_t>(k) * static_cast<size_t>(d_model) * sizeof(float)},
                         {top_w, static_cast<size_t>(k) * sizeof(float)}};
    if (any_alias(o, 1, ins, k > 0 ? 2 : 0)) return SMOE_ERR_ALIAS;
    return to_status(smoe::launch_combine(k, expert_out, top_w, out, d_model, static_cast<cudaStream_t>(stream)));
}

int smoe_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (bytes == 0) return SMOE_OK;
    if (!dst || !src) return SMOE_ERR_NULL;
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) & 15u) != 0)
        return SMOE_ERR_ALIGN;
    if (overlap(Span{dst, bytes}, Span{src, bytes})) return SMOE_ERR_ALIAS;
    void *d = smoe::device_address(dst);
    const void *s = smoe::device_address(src);
    if (!d || !s) return SMOE_ERR_MEMORY;
    return to_status(smoe::launch_copy16(d, s, bytes, static_cast<cudaStream_t>(stream)));
}

int smoe_selftest_bounded_wait(int kind, void *stream)
{
    if (kind != 0 && kind != 1) return SMOE_ERR_SHAPE;
    return to_status(smoe::launch_bounded_wait_selftest(kind, static_cast<cudaStream_t>(stream)));
}

int smoe_last_device_status(void *stream)
{
    unsigned v = 0;
    if (smoe::read_and_clear_device_status(static_cast<cudaStream_t>(stream), &v) != cudaSuccess)
        return SMOE_ERR_LAUNCH;
    if (v == smoe::kStatusRoute) return SMOE_ERR_ROUTE;
    return v ? SMOE_ERR_TIMEOUT : SMOE_OK;
}

}  // extern "C"
