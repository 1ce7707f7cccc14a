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
// Selection: every logit becomes a 64-bit key that orders (value descending,
// NaN last, index ascending) as an unsigned integer; keys are distinct.  Up
// to 256 experts, one thread per expert counts the keys above its own (its
// rank) and the k first ranks write themselves out: no rounds, two barriers.
// Above that, one CTA takes k rounds of a block-wide maximum, retiring each
// winner.
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

// The logit a key was made from (-0 comes back as +0, any NaN as a NaN).
__device__ __forceinline__ float key_value(unsigned long long key)
{
    const uint32_t u = static_cast<uint32_t>(key >> 32);
    if (u == 1u) return __int_as_float(0x7fffffff);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
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

// Softmax over the k selected logits sel_v[0 .. k-1] (sel_v[0] the largest)
// by warp 0, with the indices: k <= 64, so lane l takes ranks l and l + 32.
__device__ __forceinline__ void write_weights(const float *sel_v, const int *sel_e, int k, int *__restrict__ idx,
                                              float *__restrict__ w)
{
    const int t = threadIdx.x;
    const float v0 = sel_v[0];
    const float e0 = t < k ? expf(sel_v[t] - v0) : 0.f;
    const float e1 = t + 32 < k ? expf(sel_v[t + 32] - v0) : 0.f;
    float sum = e0 + e1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(FULL_MASK, sum, off);
    if (t < k) {
        idx[t] = sel_e[t];
        w[t] = e0 / sum;
    }
    if (t + 32 < k) {
        idx[t + 32] = sel_e[t + 32];
        w[t + 32] = e1 / sum;
    }
}

constexpr int TOPK_COUNT_MAX = 256;

// n <= 256: thread e's rank is the number of keys above its own.
__global__ void __launch_bounds__(TOPK_COUNT_MAX) topk_count(const float *__restrict__ logits, int n, int k,
                                                             int *__restrict__ idx, float *__restrict__ w)
{
    __shared__ __align__(16) unsigned long long keys[TOPK_COUNT_MAX];
    __shared__ float sel_v[SMOE_MAX_TOP_K];
    __shared__ int sel_e[SMOE_MAX_TOP_K];
    const int t = threadIdx.x;
    pdl_wait();  // the logits come from the previous kernel
    const float v = t < n ? logits[t] : 0.f;
    const unsigned long long mine = t < n ? rank_key(v, t) : 0ull;  // 0: below every key
    keys[t] = mine;
    __syncthreads();
    pdl_launch_dependents();
    if (t < n) {
        const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(keys);
        int rank = 0;
        for (int j = 0; j < (n + 1) >> 1; ++j) {  // keys[n] (odd n) is a 0 pad
            const ulonglong2 p = k2[j];
            rank += (p.x > mine) + (p.y > mine);
        }
        if (rank < k) {
            sel_v[rank] = v;
            sel_e[rank] = t;
        }
    }
    __syncthreads();
    if (t < 32) write_weights(sel_v, sel_e, k, idx, w);
}

__global__ void __launch_bounds__(TOPK_THREADS) topk_weights(const float *__restrict__ logits, int n, int k,
                                                             int *__restrict__ idx, float *__restrict__ w)
{
    extern __shared__ unsigned long long keys[];  // [n]
    __shared__ unsigned long long warp_best[TOPK_THREADS / 32];
    __shared__ int chosen[SMOE_MAX_TOP_K];
    __shared__ float chosen_v[SMOE_MAX_TOP_K];
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
                chosen_v[r] = key_value(b);
                keys[e] = 0;  // retired
            }
        }
        __syncthreads();
    }
    pdl_launch_dependents();
    if (t < 32) write_weights(chosen_v, chosen, k, idx, w);
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
    if (n_experts <= TOPK_COUNT_MAX)
        return launch_pdl(topk_count, dim3(1), dim3(TOPK_COUNT_MAX), 0, stream, logits, n_experts, k, idx, w);
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
