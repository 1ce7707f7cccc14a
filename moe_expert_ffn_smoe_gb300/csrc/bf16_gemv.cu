// Dense bf16 matvec y = W x (f32 x and y), the S-MoE page "Metal Compute
// Kernels", section "Coalesced Dense Matvec -- the Same Contract for bf16".
//
// GB300 layout: a CTA owns a contiguous block of rows (the blocks differ by
// at most one row) and all its 512 threads work on every row together:
// thread t reads the 16-byte chunks t, t + 512, ... (8 bf16 each) of the
// row, so every row is one fully coalesced sweep and no warp idles while
// others finish.  Rows are processed in groups of G (8 / chunks per
// thread, at least 2): the loads of the next group are in flight while the
// current group is multiplied.  x is staged in shared memory once per CTA;
// for rows of up to 8192 columns each thread keeps the x values of its
// chunks in registers.  A bf16 is the upper half of an f32, so widening is
// a shift or a mask.  Per row, the 512 partial sums are reduced with warp
// shuffles and one shared-memory step.  The CTA prefetches the head of its
// row block into L2 before waiting on the previous kernel.
//
// Batched form (section "Batched Scout Matvec": N independent matvecs in one
// submission): one grid of about one CTA per SM is shared by the matvecs in
// proportion to their weight bytes, each CTA running the same row-block
// sweep on its matvec, so many small matvecs cost one launch ramp.
#include "bf16_rows.cuh"
#include "common.cuh"
#include "internal.h"

namespace smoe {

struct Bf16Args {
    const uint16_t *w;
    const float *x;
    float *y;
    int rows;
    int K;
    uint32_t prefetch_bytes;  // per CTA, from the start of its row block
};

// N independent matvecs in one grid ("Batched Scout Matvec"): matvec i owns
// CTAs [cta0[i], cta0[i + 1]), each a contiguous block of its rows.  All
// matvecs of one launch take the same chunks per thread (CPL).
constexpr int BF_BATCH_MAX = 64;

struct Bf16BatchArgs {
    const uint16_t *w[BF_BATCH_MAX];
    const float *x[BF_BATCH_MAX];
    float *y[BF_BATCH_MAX];
    int rows[BF_BATCH_MAX];
    int K[BF_BATCH_MAX];
    int cta0[BF_BATCH_MAX + 1];
    int n;
    uint32_t prefetch_bytes;
};

template <int CPL>
__global__ void __launch_bounds__(BF_THREADS, 1) bf16_gemv(Bf16Args a)
{
    extern __shared__ __align__(16) float4 xs[];
    __shared__ float part[2][BF_WARPS][BF_GMAX];
    const int r0 = static_cast<int>(static_cast<long long>(a.rows) * blockIdx.x / gridDim.x);
    const int r1 = static_cast<int>(static_cast<long long>(a.rows) * (blockIdx.x + 1) / gridDim.x);
    bf16_rows<CPL>(a.w, a.x, a.y, r0, r1, a.K, a.prefetch_bytes, xs, part);
}

template <int CPL>
__global__ void __launch_bounds__(BF_THREADS, 1) bf16_gemv_batch(const __grid_constant__ Bf16BatchArgs a)
{
    extern __shared__ __align__(16) float4 xs[];
    __shared__ float part[2][BF_WARPS][BF_GMAX];
    // the matvec this CTA belongs to: the last i with cta0[i] <= blockIdx.x
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cta0[mid] <= static_cast<int>(blockIdx.x)) lo = mid;
        else hi = mid - 1;
    }
    const int i = lo;
    const int nb = a.cta0[i + 1] - a.cta0[i];
    const int b = static_cast<int>(blockIdx.x) - a.cta0[i];
    const int r0 = static_cast<int>(static_cast<long long>(a.rows[i]) * b / nb);
    const int r1 = static_cast<int>(static_cast<long long>(a.rows[i]) * (b + 1) / nb);
    bf16_rows<CPL>(a.w[i], a.x[i], a.y[i], r0, r1, a.K[i], a.prefetch_bytes, xs, part);
}

cudaError_t launch_bf16_gemv(const uint16_t *w, const float *x, float *y, int rows, int K,
                             cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    Bf16Args a = {w, x, y, rows, K, 0};
    const int KC = K / 8;
    int cpl = (KC + BF_THREADS - 1) / BF_THREADS;
    if (cpl < 1) cpl = 1;  // K = 0: every chunk reads as zero, y = 0
    const size_t smem = static_cast<size_t>(K > 0 ? K : 4) * sizeof(float);
    long long grid = dev->sm_count;
    if (rows < grid) grid = rows < 1 ? 1 : rows;
    // Prefetch at most 1/4 of L2's worth across the grid.
    const size_t l2_share = static_cast<size_t>(32u << 20) / static_cast<size_t>(grid);
    a.prefetch_bytes = static_cast<uint32_t>(l2_share < (1u << 20) ? l2_share : (1u << 20));
    void (*k)(Bf16Args) = nullptr;
    switch (cpl) {
    case 1: k = bf16_gemv<1>; break;
    case 2: k = bf16_gemv<2>; break;
    case 3: k = bf16_gemv<3>; break;
    case 4: k = bf16_gemv<4>; break;
    case 5: k = bf16_gemv<5>; break;
    case 6: k = bf16_gemv<6>; break;
    case 7: k = bf16_gemv<7>; break;
    case 8: k = bf16_gemv<8>; break;
    default: return cudaErrorInvalidValue;  // K > SMOE_MAX_COLS is refused earlier
    }
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(static_cast<unsigned>(grid)), dim3(BF_THREADS), smem, stream, a);
}

namespace {

int bf16_cpl(int K)
{
    const int cpl = (K / 8 + BF_THREADS - 1) / BF_THREADS;
    return cpl < 1 ? 1 : cpl;
}

using BatchKernel = void (*)(Bf16BatchArgs);

BatchKernel batch_kernel(int cpl)
{
    switch (cpl) {
    case 1: return bf16_gemv_batch<1>;
    case 2: return bf16_gemv_batch<2>;
    case 3: return bf16_gemv_batch<3>;
    case 4: return bf16_gemv_batch<4>;
    case 5: return bf16_gemv_batch<5>;
    case 6: return bf16_gemv_batch<6>;
    case 7: return bf16_gemv_batch<7>;
    case 8: return bf16_gemv_batch<8>;
    default: return nullptr;
    }
}

// One launch for entries idx[0..cnt) (same CPL, rows > 0): about one CTA per
// SM in total, split over the matvecs in proportion to their weight bytes,
// at least one CTA each and never more CTAs than rows.
cudaError_t launch_batch_part(const uint16_t *const *w, const float *const *x, float *const *y, const int *rows,
                              const int *cols, const int *idx, int cnt, int cpl, int sm_count, cudaStream_t stream)
{
    Bf16BatchArgs a = {};
    a.n = cnt;
    double total = 0.0;
    int kmax = 4;
    for (int j = 0; j < cnt; ++j) {
        total += static_cast<double>(rows[idx[j]]) * (cols[idx[j]] > 0 ? cols[idx[j]] : 8);
        if (cols[idx[j]] > kmax) kmax = cols[idx[j]];
    }
    int next = 0;
    for (int j = 0; j < cnt; ++j) {
        const int i = idx[j];
        const double share = static_cast<double>(rows[i]) * (cols[i] > 0 ? cols[i] : 8) / total;
        long long nb = static_cast<long long>(share * sm_count + 0.5);
        if (nb < 1) nb = 1;
        if (nb > rows[i]) nb = rows[i];
        a.w[j] = w[i];
        a.x[j] = x[i];
        a.y[j] = y[i];
        a.rows[j] = rows[i];
        a.K[j] = cols[i];
        a.cta0[j] = next;
        next += static_cast<int>(nb);
    }
    a.cta0[cnt] = next;
    const size_t l2_share = static_cast<size_t>(32u << 20) / static_cast<size_t>(next);
    a.prefetch_bytes = static_cast<uint32_t>(l2_share < (1u << 20) ? l2_share : (1u << 20));
    BatchKernel k = batch_kernel(cpl);
    if (!k) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kmax) * sizeof(float);
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(static_cast<unsigned>(next)), dim3(BF_THREADS), smem, stream, a);
}

}  // namespace

cudaError_t launch_bf16_gemv_batch(int n, const uint16_t *const *w, const float *const *x, float *const *y,
                                   const int *rows, const int *cols, cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    // one launch per chunks-per-thread class present, 64 matvecs at most each
    for (int cpl = 1; cpl <= 8; ++cpl) {
        int idx[BF_BATCH_MAX];
        int cnt = 0;
        for (int i = 0; i < n; ++i) {
            if (rows[i] == 0 || bf16_cpl(cols[i]) != cpl) continue;
            idx[cnt++] = i;
            if (cnt == BF_BATCH_MAX) {
                cudaError_t e = launch_batch_part(w, x, y, rows, cols, idx, cnt, cpl, dev->sm_count, stream);
                if (e != cudaSuccess) return e;
                cnt = 0;
            }
        }
        if (cnt > 0) {
            cudaError_t e = launch_batch_part(w, x, y, rows, cols, idx, cnt, cpl, dev->sm_count, stream);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace smoe
