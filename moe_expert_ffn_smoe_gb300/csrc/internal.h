// Host-side interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace smoe {

struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;  // largest dynamic shared memory one block may opt into
};

// Properties of the current device, cached per device; nullptr if the
// device cannot be queried.
const DeviceInfo *device_info();

// Launches y = W x for `units` output rows of a packed Q4/Q2 matrix, or the
// fused gate/up pass when nmat == 2 (codes[0]/scales[0] = gate,
// codes[1]/scales[1] = up, y = hidden).  Shapes are already validated.
cudaError_t launch_qgemv(int bits, int nmat, const uint8_t *const codes[2],
                         const float *const scales[2], const float *x, float *y,
                         int units, int K, int group, cudaStream_t stream);

// Bulk-copy + integer-dot decode kernel over n_experts experts at once
// (one grid slice per expert).  codes1/scales1 are used when nmat == 2.
// x[e], y[e] are expert e's input and output.  Sets *unsupported (and
// launches nothing) for shapes this kernel does not take.
cudaError_t launch_qgemv_experts(int bits, int nmat, int n_experts, const uint8_t *const *codes0,
                                 const uint8_t *const *codes1, const float *const *scales0,
                                 const float *const *scales1, const float *const *x, float *const *y,
                                 int units, int K, int group, cudaStream_t stream, bool *unsupported);

// The same kernels for a routed launch: slot e (of n_slots <= 64) uses the
// weights of expert route[e] (a device array written by an earlier kernel)
// from device tables of n_route pointers; x[e], y[e] are the slot's input
// and output.  Sets *unsupported (and launches nothing) for shapes these
// kernels do not take.
cudaError_t launch_qgemv_routed(int bits, int nmat, int n_slots, const uint8_t *const *tab_codes0,
                                const uint8_t *const *tab_codes1, const float *const *tab_scales0,
                                const float *const *tab_scales1, const int *route, int n_route,
                                const float *const *x, float *const *y, int units, int K, int group,
                                cudaStream_t stream, bool *unsupported);

// Device status word value of a routed index outside its table.
constexpr unsigned kStatusRoute = 16u;

// The fused routed-expert FFN over n <= 64 experts in one launch
// (expert_ffn.cu): hidden [n x d_ff] and the hand-off counters `sync`
// (2 x 64 words, zero on entry, zero again on completion) live in the
// caller's workspace.  Sets *unsupported (and launches nothing) for shapes
// the fused kernel does not take.
cudaError_t launch_expert_ffn(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                              const uint8_t *const *uc, const float *const *us, const uint8_t *const *dc,
                              const float *const *ds, const float *x, float *hidden, float *out, unsigned *sync,
                              int d_model, int d_ff, int group, cudaStream_t stream, bool *unsupported);

// Device address of the library's device status word on the current device.
unsigned *device_status_word();

// Launches y = W x for a bf16 [rows x K] matrix.  Shapes already validated.
cudaError_t launch_bf16_gemv(const uint16_t *w, const float *x, float *y, int rows, int K,
                             cudaStream_t stream);

// n independent bf16 matvecs (host arrays of device pointers and sizes,
// checked by the caller); entries with rows == 0 are skipped.
cudaError_t launch_bf16_gemv_batch(int n, const uint16_t *const *w, const float *const *x, float *const *y,
                                   const int *rows, const int *cols, cudaStream_t stream);

// Router logits (bf16 matvec), then top-k indices and weights (route.cu).
cudaError_t launch_route(const uint16_t *gate_w, const float *x, int n_experts, int d_model, int k, float *logits,
                         int *idx, float *w, cudaStream_t stream);
// out = sum_i w[i] eo[i] over k rows of d_model (route.cu).
cudaError_t launch_combine(int k, const float *eo, const float *w, float *out, int d_model, cudaStream_t stream);

// Token batch: Y[T x units] = W X^T for T tokens (nmat == 2: fused gate/up,
// Y = hidden).  Shapes already validated.
cudaError_t launch_qgemm_tokens(int bits, int nmat, const uint8_t *const codes[2],
                                const float *const scales[2], const float *X, float *Y,
                                int T, int units, int K, int group, cudaStream_t stream);

// Tensor-core batch path (ffn_batch_tc.cu): shapes it takes, its workspace,
// and the launch of its four kernels (operand preparation and GEMM for
// gate/up, then for down).
bool tc_batch_supported(int T, int d_model, int d_ff, int group);
bool tc_batch_shape_supported(int d_model, int d_ff, int group);
size_t tc_batch_workspace(int T, int d_model, int d_ff);
// Token batches of n experts (expert e: T[e] tokens, T[e] == 0 skipped) on
// the tensor cores in one launch set per 32 experts; shapes already checked.
size_t tc_batch_workspace_experts(int n, const int *T, int d_model, int d_ff);
cudaError_t launch_ffn_batch_tc_experts(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                                        const uint8_t *const *uc, const float *const *us,
                                        const uint8_t *const *dc, const float *const *ds,
                                        const float *const *X, float *const *Y, const int *T, int d_model,
                                        int d_ff, int group, void *workspace, cudaStream_t stream);
cudaError_t launch_ffn_batch_tc(int bits, const uint8_t *const gu_codes[2], const float *const gu_scales[2],
                                const uint8_t *down_codes, const float *down_scales, const float *X, float *Y,
                                int T, int d_model, int d_ff, int group, void *workspace, cudaStream_t stream);

// Bytes of workspace the batch FFN needs (0 for T <= 0).
size_t ffn_batch_workspace(int T, int d_model, int d_ff, int group);

// The whole batch FFN: gate/up into the workspace, then down into Y.
cudaError_t launch_ffn_batch(int bits, const uint8_t *const gu_codes[2], const float *const gu_scales[2],
                             const uint8_t *down_codes, const float *down_scales,
                             const float *X, float *Y, int T, int d_model, int d_ff, int group,
                             void *workspace, cudaStream_t stream);

// Token batches of n experts: the grouped tensor-core launches when the
// shape allows, else expert after expert through launch_ffn_batch.
size_t ffn_batch_workspace_experts(int n, const int *T, int d_model, int d_ff, int group);
cudaError_t launch_ffn_batch_experts(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                                     const uint8_t *const *uc, const float *const *us,
                                     const uint8_t *const *dc, const float *const *ds, const float *const *X,
                                     float *const *Y, const int *T, int d_model, int d_ff, int group,
                                     void *workspace, cudaStream_t stream);

// Reads and clears the device status word of the current device after
// synchronising `stream`.
cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned *value);
// dst[0 .. bytes) = src[0 .. bytes), both device addresses, 16-byte aligned,
// bytes a multiple of 16, by the SMs (copy.cu).
cudaError_t launch_copy16(void *dst, const void *src, size_t bytes, cudaStream_t stream);
// Device address of a device-accessible buffer, null for pageable host
// memory or an unknown pointer (copy.cu).
void *device_address(const void *p);

// One warp whose bounded wait never succeeds (kind 0: an mbarrier, kind 1:
// a device counter); it records a timeout in the status word (selftest.cu).
cudaError_t launch_bounded_wait_selftest(int kind, cudaStream_t stream);

// cudaLaunchKernelEx with programmatic dependent launch enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_pdl as a cooperative launch: CUDA starts the grid only when all of
// its CTAs can be resident at once (and refuses a grid that never could),
// which a kernel whose CTAs wait on one another needs.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_pdl with thread-block clusters of (1, 1, cluster_z) CTAs
// (cluster_z == 1: no cluster attribute).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_z, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = cluster_z;
    cfg.attrs = attr;
    cfg.numAttrs = cluster_z > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Opts a kernel into `bytes` of dynamic shared memory.  Static shared memory
// counts against the default 48 KB too, so the limit is raised for any
// nonzero size it does not already cover.  It is only ever raised: one
// kernel serves launches of different shared-memory sizes, and a launch
// captured earlier into a graph must stay valid after a later, smaller
// launch of the same kernel.
template <typename K>
cudaError_t ensure_dynamic_smem(K kernel, size_t bytes)
{
    if (bytes == 0) return cudaSuccess;
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kernel));
    if (err != cudaSuccess) return err;
    if (static_cast<size_t>(fa.maxDynamicSharedSizeBytes) >= bytes) return cudaSuccess;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel),
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

}  // namespace smoe
