// Routing and the weighted combine of a token's expert outputs.
//
// The S-MoE page "Metal Compute Kernels" runs the exact-routing gate matvec
// (n_experts x d_model) on the host ("Batched Scout Matvec") and describes
// neither the selection nor the weighting.  The readings implemented here:
//   logits = G x, G in bf16 (the dense matvec of bf16_gemv.cu);
//   the k largest logits in descending order, ties to the lower expert
//     index, NaN below every number;
//   weights: exp(l_i - l_max) / sum over the k selected of exp(l_j - l_max);
//   out[j] = sum over the k selected, in selection order, of w_i y_i[j].
//
// Selection: one CTA keeps every logit as a 64-bit key that orders (value
// descending, NaN last, index ascending) as an unsigned integer, and takes k
// rounds of a block-wide maximum, retiring each winner.
#include "common.cuh"
#include "internal.h"
#include "smoe.h"

namespace smoe {

namespace {

constexpr int TOPK_THREADS = 256;

// Order-preserving key: larger key = ranks first.
__device__ __forceinline__ unsigned long long rank_key(float v, int e)
{
    uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);  // -0 ranks with +0 (ties by index)
    if (isnan(v)) u = 1u;  // above a retired slot (0), below every number (-inf maps to 0x007FFFFF)
    else u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(FULL_MASK, k, off);
        k = o > k ? o : k;
    }
    return k;
}

__global__ void __launch_bounds__(TOPK_THREADS) topk_weights(const float *__restrict__ logits, int n, int k,
                                                             int *__restrict__ idx, float *__restrict__ w)
{
    extern __shared__ unsigned long long keys[];  // [n]
    __shared__ unsigned long long warp_best[TOPK_THREADS / 32];
    __shared__ int chosen[SMOE_MAX_TOP_K];
    const int t = threadIdx.x;
    pdl_wait();  // the logits come from the previous kernel
    for (int e = t; e < n; e += TOPK_THREADS) keys[e] = rank_key(logits[e], e);
    __syncthreads();
    for (int r = 0; r < k; ++r) {
        unsigned long long best = 0;
        for (int e = t; e < n; e += TOPK_THREADS) best = keys[e] > best ? keys[e] : best;
        best = warp_max_u64(best);
        if ((t & 31) == 0) warp_best[t >> 5] = best;
        __syncthreads();
        if (t < 32) {
            unsigned long long b = t < TOPK_THREADS / 32 ? warp_best[t] : 0;
            b = warp_max_u64(b);
            if (t == 0) {
                const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(b));
                chosen[r] = e;
                keys[e] = 0;  // retired
            }
        }
        __syncthreads();
    }
    pdl_launch_dependents();
    if (t == 0) {
        const float lmax = logits[chosen[0]];
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += expf(logits[chosen[r]] - lmax);
        for (int r = 0; r < k; ++r) {
            idx[r] = chosen[r];
            w[r] = expf(logits[chosen[r]] - lmax) / sum;
        }
    }
}

// out[j] = sum_i w[i] * eo[i][j], i in selection order.
__global__ void __launch_bounds__(256) combine_rows(const float *__restrict__ eo, const float *__restrict__ w,
                                                    int k, float *__restrict__ out, int d_model)
{
    pdl_wait();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < d_model) {
        float acc = 0.f;
        for (int i = 0; i < k; ++i) acc = fmaf(w[i], eo[static_cast<size_t>(i) * d_model + j], acc);
        out[j] = acc;
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const uint16_t *gate_w, const float *x, int n_experts, int d_model, int k, float *logits,
                         int *idx, float *w, cudaStream_t stream)
{
    cudaError_t e = launch_bf16_gemv(gate_w, x, logits, n_experts, d_model, stream);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(n_experts) * sizeof(unsigned long long);
    e = ensure_dynamic_smem(topk_weights, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_weights, dim3(1), dim3(TOPK_THREADS), smem, stream, logits, n_experts, k, idx, w);
}

cudaError_t launch_combine(int k, const float *eo, const float *w, float *out, int d_model, cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>((d_model + 255) / 256);
    return launch_pdl(combine_rows, dim3(blocks), dim3(256), 0, stream, eo, w, k, out, d_model);
}

}  // namespace smoe
