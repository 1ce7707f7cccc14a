// Token-batch fused FFN of one Q4 expert, the S-MoE page "Metal Compute
// Kernels", section "Token-Batch Fused FFN": the one-token FFN applied to
// every row of X [T x d_model], gate/up+SiLU into H [T x d_ff] (the caller's
// workspace), then down into Y [T x d_model].
//
// Paths: one token goes through the decode kernels (qgemv.cu); 2 to 6
// tokens (8 where the tensor cores do not take the shape) go through the
// grouped decode kernels with one slot per token
// (qgemv_tma.cu / qgemv_reg.cu) when both row lengths are whole multiples of
// 8 chunks; more tokens go to the tensor cores (ffn_batch_tc.cu) when the
// group size and both dimensions are multiples of 64; other shapes use the
// CUDA-core multi-token GEMV below, in which a warp unpacks each 16-byte
// chunk of codes once and applies it to TT tokens whose x rows are staged in
// shared memory.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "qformat.cuh"

namespace smoe {

// Device status word: set by device-side bounded waits that gave up.
__device__ unsigned int g_device_status = 0;

struct QTokArgs {
    const uint8_t *codes[2];
    const float *scales[2];
    const float *X;  // [T x K]
    float *Y;        // [T x units]
    int T;
    int units;
    int K;
    int group;
};

template <int BITS, int NMAT, int TT>
__global__ void __launch_bounds__(256) qgemm_tokens(QTokArgs a)
{
    using F = QFmt<BITS>;
    constexpr int F4W = F::CODES_PER_WORD / 4;
    extern __shared__ __align__(16) float4 smem4[];
    const int KC = a.K / F::CODES_PER_CHUNK;
    const int nq = a.K >> 2;
    float4 *xs = smem4;  // [TT][nq]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int ngroups = a.K / a.group;
    const int cpg = a.group / F::CODES_PER_CHUNK;
    const size_t row_bytes = static_cast<size_t>(KC) * 16;

    pdl_wait();

    const uint32_t xs_base = smem_addr(xs);
    uint32_t xo[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) xo[m] = static_cast<uint32_t>(m ^ (lane & 7)) * 16u;

    for (int tb = blockIdx.y * TT; tb < a.T; tb += gridDim.y * TT) {
        __syncthreads();  // the previous tile's readers are done
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const int tok = tb + t < a.T ? tb + t : a.T - 1;  // repeat the last token as padding
            stage_x_chunks<BITS>(a.X + static_cast<size_t>(tok) * a.K, a.K, xs + static_cast<size_t>(t) * nq);
        }
        __syncthreads();

        for (int unit = blockIdx.x * nwarps + warp; unit < a.units; unit += gridDim.x * nwarps) {
            float acc[NMAT][TT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int t = 0; t < TT; ++t) acc[m][t] = 0.f;

            for (int cc = lane; cc < KC; cc += 32) {
                uint4 cw[NMAT];
                float sc[NMAT];
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    cw[m] = ldg_stream(a.codes[m] + unit * row_bytes + static_cast<size_t>(cc) * 16);
                    sc[m] = ldg_f32(a.scales[m] + static_cast<size_t>(unit) * ngroups + cc / cpg);
                }
                float P[NMAT][TT];
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int t = 0; t < TT; ++t) P[m][t] = 0.f;
                const uint32_t cbase = xs_base + static_cast<uint32_t>(cc * F::F4_PER_CHUNK) * 16u;
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    float f[NMAT][F::CODES_PER_WORD];
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint32_t w = word_of(cw[m], wi);
#pragma unroll
                        for (int i = 0; i < F::CODES_PER_WORD; ++i) f[m][i] = code_centred<BITS>(w, i);
                    }
#pragma unroll
                    for (int t = 0; t < TT; ++t) {
                        const uint32_t tbase = cbase + static_cast<uint32_t>(t) * static_cast<uint32_t>(nq) * 16u;
#pragma unroll
                        for (int q = 0; q < F4W; ++q) {
                            const int mq = wi * F4W + q;
                            const float4 v = lds128(tbase + static_cast<uint32_t>((mq & 8) * 16) + xo[mq & 7]);
#pragma unroll
                            for (int m = 0; m < NMAT; ++m) {
                                P[m][t] = fmaf(f[m][4 * q + 0], v.x, P[m][t]);
                                P[m][t] = fmaf(f[m][4 * q + 1], v.y, P[m][t]);
                                P[m][t] = fmaf(f[m][4 * q + 2], v.z, P[m][t]);
                                P[m][t] = fmaf(f[m][4 * q + 3], v.w, P[m][t]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < TT; ++t)
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) acc[m][t] = fmaf(sc[m], P[m][t], acc[m][t]);
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int t = 0; t < TT; ++t)
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) acc[m][t] += __shfl_xor_sync(FULL_MASK, acc[m][t], off);
            if (lane == 0) {
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    if (tb + t < a.T) {
                        const float y0 = F::A * acc[0][t];
                        float out = y0;
                        if (NMAT == 2) {
                            const float y1 = F::A * acc[NMAT - 1][t];
                            out = silu_f32(y0) * y1;
                        }
                        a.Y[static_cast<size_t>(tb + t) * a.units + unit] = out;
                    }
                }
            }
        }
    }
    pdl_launch_dependents();
}

namespace {

template <int BITS, int NMAT, int TT>
cudaError_t launch_tok(const QTokArgs &a, cudaStream_t stream)
{
    using F = QFmt<BITS>;
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const int KC = a.K / F::CODES_PER_CHUNK;
    const size_t smem = static_cast<size_t>(TT) * static_cast<size_t>(a.K) * sizeof(float);
    if (smem > static_cast<size_t>(dev->max_smem_optin)) return cudaErrorInvalidValue;
    const int warps = 8;
    long long gx = (static_cast<long long>(a.units) + warps - 1) / warps;
    const int tiles = (a.T + TT - 1) / TT;
    long long gy = tiles < 65535 ? tiles : 65535;
    const long long cap = static_cast<long long>(dev->sm_count) * 2;
    if (gx * gy > cap * 8 && gx > cap) gx = cap;
    auto k = qgemm_tokens<BITS, NMAT, TT>;
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(warps * 32),
                      smem, stream, a);
}

template <int NMAT>
cudaError_t launch_tok_pick(const QTokArgs &a, cudaStream_t stream)
{
    // Token tile: enough tokens to amortise the unpack, few enough that the
    // x rows of a tile fit in shared memory.
    const size_t per_token = (static_cast<size_t>(a.K) + a.K / 32) * sizeof(float);
    if (a.T >= 8 && per_token * 8 <= 200 * 1024) return launch_tok<4, NMAT, 8>(a, stream);
    if (a.T >= 4 && per_token * 4 <= 200 * 1024) return launch_tok<4, NMAT, 4>(a, stream);
    if (a.T >= 2 && per_token * 2 <= 200 * 1024) return launch_tok<4, NMAT, 2>(a, stream);
    return launch_tok<4, NMAT, 1>(a, stream);
}

}  // namespace

cudaError_t launch_qgemm_tokens(int bits, int nmat, const uint8_t *const codes[2],
                                const float *const scales[2], const float *X, float *Y, int T,
                                int units, int K, int group, cudaStream_t stream)
{
    if (bits != 4) return cudaErrorInvalidValue;
    QTokArgs a = {};
    a.codes[0] = codes[0];
    a.codes[1] = nmat == 2 ? codes[1] : codes[0];
    a.scales[0] = scales[0];
    a.scales[1] = nmat == 2 ? scales[1] : scales[0];
    a.X = X;
    a.Y = Y;
    a.T = T;
    a.units = units;
    a.K = K;
    a.group = group;
    return nmat == 2 ? launch_tok_pick<2>(a, stream) : launch_tok_pick<1>(a, stream);
}

namespace {

// Token counts from 2 to kSlotTokens run as T one-token decodes of the same
// expert: the grouped decode kernels with one slot per token, all slots
// sharing the expert's weights (read from DRAM once, the other slots' reads
// hit L2).  Below the measured crossover this is faster than the tensor
// cores, whose per-call latency (token prep, first K tile, split-K finish)
// does not shrink with T: one expert at d_model 4096, d_ff 1536 took
// 16.5 / 18.4 us (slots, T = 6 / 7) against 17.6 / 17.6 us (tensor cores).
// Shapes the tensor cores do not take keep the slots up to kSlotTokensMax.
constexpr int kSlotTokens = 6;
constexpr int kSlotTokensMax = 8;

// Shapes the grouped decode kernels take for both projections: rows of
// whole multiples of 8 chunks of 16 bytes, at most 8192 columns.
bool slot_path(int bits, int T, int d_model, int d_ff, int group)
{
    const int unit = bits == 4 ? 256 : 512;
    if (T < 2 || T > kSlotTokensMax || d_model <= 0 || d_ff <= 0 || d_model % unit || d_ff % unit ||
        d_model > 8192 || d_ff > 8192)
        return false;
    return T <= kSlotTokens || !tc_batch_supported(T, d_model, d_ff, group);
}

}  // namespace

size_t ffn_batch_workspace(int T, int d_model, int d_ff, int group)
{
    if (T <= 0) return 0;
    // the slot path and the CUDA-core path need hidden f32 [T x d_ff]; the
    // size does not depend on the code width, so a token count that a Q4
    // call runs on the slots while a Q2 call of the same shape takes the
    // tensor cores gets the larger of the two
    const size_t hidden = (static_cast<size_t>(T) * static_cast<size_t>(d_ff) * sizeof(float) + 255) &
                          ~static_cast<size_t>(255);
    if (T > 1 && tc_batch_supported(T, d_model, d_ff, group)) {
        const size_t tc = tc_batch_workspace(T, d_model, d_ff);
        return tc > hidden ? tc : hidden;
    }
    return hidden;
}

cudaError_t launch_ffn_batch(int bits, const uint8_t *const gu_codes[2], const float *const gu_scales[2],
                             const uint8_t *down_codes, const float *down_scales, const float *X,
                             float *Y, int T, int d_model, int d_ff, int group, void *workspace,
                             cudaStream_t stream)
{
    float *H = static_cast<float *>(workspace);
    const uint8_t *dc[2] = {down_codes, down_codes};
    const float *ds[2] = {down_scales, down_scales};
    cudaError_t e = cudaSuccess;
    if (T == 1) {
        if (d_ff > 0) e = launch_qgemv(bits, 2, gu_codes, gu_scales, X, H, d_ff, d_model, group, stream);
        if (e != cudaSuccess) return e;
        return launch_qgemv(bits, 1, dc, ds, H, Y, d_model, d_ff, group, stream);
    }
    if (slot_path(bits, T, d_model, d_ff, group)) {
        const uint8_t *c0[kSlotTokensMax], *c1[kSlotTokensMax];
        const float *s0[kSlotTokensMax], *s1[kSlotTokensMax], *xs[kSlotTokensMax];
        float *ys[kSlotTokensMax];
        for (int t = 0; t < T; ++t) {
            c0[t] = gu_codes[0];
            c1[t] = gu_codes[1];
            s0[t] = gu_scales[0];
            s1[t] = gu_scales[1];
            xs[t] = X + static_cast<size_t>(t) * d_model;
            ys[t] = H + static_cast<size_t>(t) * d_ff;
        }
        bool unsupported = true;
        e = launch_qgemv_experts(bits, 2, T, c0, c1, s0, s1, xs, ys, d_ff, d_model, group, stream, &unsupported);
        if (e != cudaSuccess || unsupported) return unsupported ? cudaErrorInvalidValue : e;
        for (int t = 0; t < T; ++t) {
            c0[t] = down_codes;
            s0[t] = down_scales;
            xs[t] = H + static_cast<size_t>(t) * d_ff;
            ys[t] = Y + static_cast<size_t>(t) * d_model;
        }
        e = launch_qgemv_experts(bits, 1, T, c0, c0, s0, s0, xs, ys, d_model, d_ff, group, stream, &unsupported);
        return unsupported ? cudaErrorInvalidValue : e;
    }
    if (tc_batch_supported(T, d_model, d_ff, group))
        return launch_ffn_batch_tc(bits, gu_codes, gu_scales, down_codes, down_scales, X, Y, T, d_model, d_ff,
                                   group, workspace, stream);
    // Q2 shapes (columns and groups multiples of 64) always take the
    // tensor cores unless d_ff == 0, where Y = 0 and no code is read
    if (bits != 4 && d_ff > 0) return cudaErrorInvalidValue;
    if (d_ff > 0)
        e = launch_qgemm_tokens(4, 2, gu_codes, gu_scales, X, H, T, d_ff, d_model, group, stream);
    if (e != cudaSuccess) return e;
    return launch_qgemm_tokens(4, 1, dc, ds, H, Y, T, d_model, d_ff, group, stream);
}

size_t ffn_batch_workspace_experts(int n, const int *T, int d_model, int d_ff, int group)
{
    if (tc_batch_shape_supported(d_model, d_ff, group)) return tc_batch_workspace_experts(n, T, d_model, d_ff);
    size_t need = 0;
    for (int e = 0; e < n; ++e) {
        const size_t w = ffn_batch_workspace(T[e], d_model, d_ff, group);
        need = w > need ? w : need;
    }
    return need;
}

cudaError_t launch_ffn_batch_experts(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                                     const uint8_t *const *uc, const float *const *us,
                                     const uint8_t *const *dc, const float *const *ds, const float *const *X,
                                     float *const *Y, const int *T, int d_model, int d_ff, int group,
                                     void *workspace, cudaStream_t stream)
{
    if (tc_batch_shape_supported(d_model, d_ff, group))
        return launch_ffn_batch_tc_experts(bits, n, gc, gs, uc, us, dc, ds, X, Y, T, d_model, d_ff, group,
                                           workspace, stream);
    // one expert after another; each call's kernels finish reading the
    // workspace before the next call's first kernel writes it (stream order)
    for (int e = 0; e < n; ++e) {
        if (T[e] <= 0) continue;
        const uint8_t *guc[2] = {gc[e], uc[e]};
        const float *gus[2] = {gs[e], us[e]};
        cudaError_t err = launch_ffn_batch(bits, guc, gus, dc[e], ds[e], X[e], Y[e], T[e], d_model, d_ff, group,
                                           workspace, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

unsigned *device_status_word()
{
    constexpr int kMaxDevices = 64;
    static unsigned *addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned *>(p);
    }
    return addr[dev];
}

cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned *value)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_device_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned));
}

}  // namespace smoe
