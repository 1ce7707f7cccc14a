/*
 * smoe.h -- C ABI of libsmoe.so: group-quantized matrix-vector products for
 * routed mixture-of-experts FFN layers on NVIDIA GB300 (sm_103a).
 *
 * Every operation is defined by the S-MoE documentation page
 * "Metal Compute Kernels"; each declaration names the section it follows.
 * Two support functions are not steps of that method: smoe_copy (a step's
 * host I/O) and smoe_selftest_bounded_wait (a diagnostic of the device-side
 * failure detection).
 *
 * Common conventions
 * ------------------
 * Pointers.  Every pointer argument except `stream`, the results of the
 *   query functions and the two buffers of smoe_copy (which may also be
 *   pinned host memory) is a DEVICE pointer owned by the caller.  The library
 *   allocates no memory of its own on any call and keeps no pointer after the
 *   call returns.  An OUTPUT (out, y, hidden, top_idx, ...) may also be
 *   page-locked host memory mapped into the device's address space (unified
 *   addressing, e.g. cudaHostAlloc or torch's pin_memory on a node whose GPU
 *   reaches host memory over a coherent link): the kernels then write each
 *   result over the host link once, with no copy afterwards.  Inputs must be
 *   device memory (weights, tokens and hidden vectors are read by many CTAs).
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  Calls enqueue their kernels on it and return at once;
 *   results are ready when the stream's work has completed.  Kernels are
 *   launched with programmatic dependent launch: each kernel may prefetch its
 *   WEIGHTS into L2 before the previous kernel in the stream has finished,
 *   but reads its activations and writes its outputs only after the previous
 *   kernel's writes are visible.  Weights must not be written by a kernel
 *   that is still running when the call is made on the same stream unless
 *   that kernel finishes before this call's kernel starts (ordinary stream
 *   order does this for every non-kernel operation and every kernel launched
 *   without programmatic dependent launch).
 * Packed codes.  A Q4 row of `cols` weights is cols/2 bytes: byte j holds
 *   column 2j in its low nibble and column 2j+1 in its high nibble.  A Q2 row
 *   is cols/4 bytes: byte j holds columns 4j..4j+3, the first in the lowest
 *   two bits.  Rows are stored one after another with no padding, so a
 *   [rows x cols] matrix is rows*cols*bits/8 bytes.
 * Scales.  f32, row-major [rows][cols/group]: scales[r][g] applies to columns
 *   g*group .. g*group+group-1 of row r.
 * Dequantisation.  w = (code - Z) * (1/Z) * s with Z = 7.5 (Q4) or 1.5 (Q2)
 *   ("Fused FFN Kernels -- One Simdgroup Per Output Row").
 * Layout contract ("Layout assumptions the kernels rely on"): cols is a
 *   multiple of 32 (Q4) or 64 (Q2); group is a positive multiple of 32 (Q4)
 *   or 64 (Q2) that divides cols; codes, x, hidden, out, X, Y and workspace
 *   are 16-byte aligned; scales are 16-byte aligned.  Sizes are >= 0 and
 *   cols <= SMOE_MAX_COLS.
 * Empty work.  A call whose output is empty (0 rows, or T == 0) returns
 *   SMOE_OK without launching anything and without looking at the pointers.
 *   A call with cols == 0 and rows > 0 writes zeros (an empty sum).
 * Aliasing.  Outputs must not overlap any input or each other; an overlap
 *   is refused with SMOE_ERR_ALIAS.
 * Errors.  Every contract check runs on the host before any launch and
 *   returns a status without touching the GPU.  There is no fallback to
 *   another kernel or to the CPU: a call either runs the kernels below or
 *   returns an error.  SMOE_ERR_LAUNCH reports a CUDA launch error (the CUDA
 *   error itself stays readable with cudaGetLastError()).
 * Numerics.  Sums are reassociated (lanes, warps, groups), so results are not
 *   bit-identical to a sequential sum; they agree with an exact (f64) result
 *   within 1e-4 * sum_i |w_i x_i| + 1e-6 per output element for every finite
 *   x, whatever its dynamic range.  The one-token Q4/Q2 kernels round x per
 *   16-byte chunk of codes (32 Q4 or 64 Q2 columns) to a power-of-two grid
 *   that puts the chunk's largest |x| at 2^22 steps or more, take the code x
 *   x products exactly in integers and fold the scales in f32; the rounding
 *   adds at most 5.8e-5 (Q4) or 2.3e-5 (Q2) of sum |w x| in the worst case.
 *   The batch kernels use exact weights (code - Z)/2^b times x split into
 *   two bf16 halves (tensor cores) or f32 x (CUDA cores).  Activations must
 *   be finite: a NaN or infinity in x makes the outputs that read it NaN.
 * Devices.  The library looks up, once per device, the device addresses of
 *   its own device variables (the status word, the no-allocation workspace);
 *   after cudaDeviceReset() on a device the library must not be called
 *   again on that device in the same process.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMOE_ABI_VERSION 2

/* Largest `cols` (input length) any call accepts: the input vector of a
 * call is staged whole in one SM's shared memory (f32). */
#define SMOE_MAX_COLS 32768

typedef enum smoe_status {
    SMOE_OK = 0,
    SMOE_ERR_NULL = 1,      /* a required pointer is NULL                       */
    SMOE_ERR_ALIGN = 2,     /* a pointer breaks the alignment contract          */
    SMOE_ERR_SHAPE = 3,     /* sizes break the layout contract or the limits    */
    SMOE_ERR_WORKSPACE = 4, /* workspace missing or smaller than required       */
    SMOE_ERR_LAUNCH = 5,    /* CUDA refused a launch or a device query          */
    SMOE_ERR_TIMEOUT = 6,   /* a device-side bounded wait gave up               */
    SMOE_ERR_ALIAS = 7,     /* an output overlaps an input or another output    */
    SMOE_ERR_MEMORY = 8,    /* a buffer is not accessible from the device       */
    SMOE_ERR_ROUTE = 9      /* a device-side expert index or table entry was
                               invalid (reported by smoe_last_device_status)  */
} smoe_status;

/* ABI version (SMOE_ABI_VERSION of the built library). */
int smoe_abi_version(void);

/* Static text for a status code (never NULL). */
const char *smoe_status_string(int status);

/*
 * Fused gate/up pass of one routed expert for one token
 * ("Fused FFN Kernels -- One Simdgroup Per Output Row"):
 *
 *   hidden[i] = SiLU(gate . x)[i] * (up . x)[i],  i in [0, d_ff),
 *   SiLU(v) = v / (1 + e^-v).
 *
 * gate_codes, up_codes: packed [d_ff x d_model] (Q4 or Q2), row i = output i.
 * gate_scales, up_scales: f32 [d_ff x d_model/group].
 * x: f32 [d_model].  hidden: f32 [d_ff], written.
 * Both matrices are read in one pass over a shared copy of x.
 */
int smoe_gate_up_q4(const uint8_t *gate_codes, const float *gate_scales,
                    const uint8_t *up_codes, const float *up_scales,
                    const float *x, float *hidden,
                    int d_ff, int d_model, int group, void *stream);
int smoe_gate_up_q2(const uint8_t *gate_codes, const float *gate_scales,
                    const uint8_t *up_codes, const float *up_scales,
                    const float *x, float *hidden,
                    int d_ff, int d_model, int group, void *stream);

/*
 * Down projection of one routed expert for one token
 * ("Fused FFN Kernels -- One Simdgroup Per Output Row"):
 *
 *   out[j] = (down . hidden)[j],  j in [0, d_model).
 *
 * down_codes: packed [d_model x d_ff], grouped along d_ff.
 * down_scales: f32 [d_model x d_ff/group].  hidden: f32 [d_ff].
 * out: f32 [d_model], written.
 */
int smoe_down_q4(const uint8_t *down_codes, const float *down_scales,
                 const float *hidden, float *out,
                 int d_model, int d_ff, int group, void *stream);
int smoe_down_q2(const uint8_t *down_codes, const float *down_scales,
                 const float *hidden, float *out,
                 int d_model, int d_ff, int group, void *stream);

/*
 * Grouped expert dispatch ("Grouped Expert Dispatch"): the fused gate/up
 * pass of n_experts experts for the same token in one launch,
 *
 *   hidden[e][i] = SiLU(gate_e . x)[i] * (up_e . x)[i],  e in [0, n_experts).
 *
 * gate_codes, gate_scales, up_codes, up_scales: HOST arrays of n_experts
 * DEVICE pointers, expert e's tensors laid out as for smoe_gate_up_q4/q2
 * (all experts share d_ff, d_model and group).  x: f32 [d_model], shared
 * by all experts.  hidden: f32 [n_experts x d_ff] (expert-major), written.
 * The pointer arrays are read during the call only; the parameters travel
 * with the launch (up to 64 experts per launch), so nothing is allocated.
 * n_experts >= 0.  Each row is computed exactly as the single-expert call
 * computes it.
 */
int smoe_experts_gate_up_q4(int n_experts, const uint8_t *const *gate_codes,
                            const float *const *gate_scales,
                            const uint8_t *const *up_codes,
                            const float *const *up_scales, const float *x,
                            float *hidden, int d_ff, int d_model, int group,
                            void *stream);
int smoe_experts_gate_up_q2(int n_experts, const uint8_t *const *gate_codes,
                            const float *const *gate_scales,
                            const uint8_t *const *up_codes,
                            const float *const *up_scales, const float *x,
                            float *hidden, int d_ff, int d_model, int group,
                            void *stream);

/*
 * Grouped down projection ("Grouped Expert Dispatch"):
 *
 *   out[e][j] = (down_e . hidden[e])[j],  e in [0, n_experts).
 *
 * down_codes, down_scales: HOST arrays of n_experts DEVICE pointers (as for
 * smoe_down_q4/q2).  hidden: f32 [n_experts x d_ff]; out: f32
 * [n_experts x d_model] (expert-major), written.  Per-expert outputs are
 * kept separate: no router weighting or sum over experts is applied.
 */
int smoe_experts_down_q4(int n_experts, const uint8_t *const *down_codes,
                         const float *const *down_scales, const float *hidden,
                         float *out, int d_model, int d_ff, int group, void *stream);
int smoe_experts_down_q2(int n_experts, const uint8_t *const *down_codes,
                         const float *const *down_scales, const float *hidden,
                         float *out, int d_model, int d_ff, int group, void *stream);

/*
 * Bytes of device workspace smoe_experts_ffn_q4/q2 needs: SMOE_FFN_SYNC_BYTES
 * of hand-off counters followed by the hidden activations of up to 64
 * experts (f32 [min(n_experts, 64) x d_ff]), rounded up to 256.  Returns 0
 * for n_experts <= 0 and (size_t)-1 for d_ff < 0.
 */
#define SMOE_FFN_SYNC_BYTES 512u
size_t smoe_experts_ffn_workspace_bytes(int n_experts, int d_ff);

/*
 * The whole routed-expert FFN of one token over n_experts experts ("Fused
 * FFN Kernels -- One Simdgroup Per Output Row" for each expert, batched as
 * in "Grouped Expert Dispatch"):
 *
 *   hidden_e  = SiLU(gate_e . x) * (up_e . x)
 *   out[e][j] = (down_e . hidden_e)[j],  e in [0, n_experts).
 *
 * gate_codes ... down_scales: HOST arrays of n_experts DEVICE pointers,
 * expert e's tensors laid out as for smoe_gate_up_q4/q2 and smoe_down_q4/q2
 * (all experts share d_model, d_ff and group).  x: f32 [d_model], shared.
 * out: f32 [n_experts x d_model] (expert-major), written; no router
 * weighting or sum over experts is applied.
 * workspace: device memory of at least
 * smoe_experts_ffn_workspace_bytes(n_experts, d_ff) bytes, 16-byte aligned,
 * owned by the caller.  Its first SMOE_FFN_SYNC_BYTES must be zero before
 * the first call (one cudaMemset); every call that completes leaves them
 * zero again.  The rest holds hidden between the two halves of the call.
 * One launch covers up to 64 experts: the CTAs of an expert compute its
 * hidden rows, meet on a counter in the workspace (a bounded wait), then
 * compute its down rows, while the down weights already stream during the
 * first half.  The launch occupies one CTA per SM and assumes its CTAs run
 * together; if a wait gives up (about two seconds, e.g. when other streams
 * hold SMs for that long) the outputs are unspecified,
 * smoe_last_device_status reports SMOE_ERR_TIMEOUT and the counters must be
 * zeroed again.  Shapes the one-launch kernel does not take run as
 * smoe_experts_gate_up (into the workspace) followed by smoe_experts_down.
 * Calls that share a workspace must not overlap on the GPU.
 * Returns SMOE_ERR_WORKSPACE for a missing or short workspace and
 * SMOE_ERR_ALIAS when out, x, the workspace or any weight overlap.
 */
int smoe_experts_ffn_q4(int n_experts, const uint8_t *const *gate_codes,
                        const float *const *gate_scales,
                        const uint8_t *const *up_codes,
                        const float *const *up_scales,
                        const uint8_t *const *down_codes,
                        const float *const *down_scales, const float *x,
                        float *out, int d_model, int d_ff, int group,
                        void *workspace, size_t workspace_bytes, void *stream);
int smoe_experts_ffn_q2(int n_experts, const uint8_t *const *gate_codes,
                        const float *const *gate_scales,
                        const uint8_t *const *up_codes,
                        const float *const *up_scales,
                        const uint8_t *const *down_codes,
                        const float *const *down_scales, const float *x,
                        float *out, int d_model, int d_ff, int group,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Dense bf16 matvec ("Coalesced Dense Matvec -- the Same Contract for bf16"):
 *
 *   y[r] = sum_k bf16(w[r][k]) * x[k],  r in [0, rows).
 *
 * w: bf16 bit patterns, row-major [rows x cols], 16-byte aligned; cols is a
 * multiple of 8 (so every row starts on a 16-byte boundary) and at most
 * SMOE_MAX_COLS.  x: f32 [cols], 16-byte aligned.  y: f32 [rows], written.
 */
int matvec_bf16(const uint16_t *w, const float *x, float *y,
                int rows, int cols, void *stream);

/*
 * n independent dense bf16 matvecs in one submission ("Batched Scout
 * Matvec"):
 *
 *   y[i][r] = sum_k bf16(w[i][r][k]) * x[i][k],  i in [0, n), r in [0, rows[i]).
 *
 * w, x, y: host arrays of n device pointers; rows, cols: host arrays of n
 * sizes.  Every entry follows matvec_bf16's contract (cols[i] a multiple of 8
 * and at most SMOE_MAX_COLS, 16-byte alignment); an entry with rows[i] == 0
 * is skipped and may hold null pointers.  No output may overlap any input or
 * another output (SMOE_ERR_ALIAS).  The matvecs share one grid (one launch
 * per 64 entries of equal row-length class, usually one in all), so many
 * small matvecs pay one launch ramp.  n == 0 is a no-op.
 */
int matvec_bf16_batch(int n, const uint16_t *const *w, const float *const *x,
                      float *const *y, const int *rows, const int *cols,
                      void *stream);

/*
 * Bytes of device workspace ffn_batch_q4 and ffn_batch_q2 need for these
 * sizes (the token operand and the hidden activations in the tensor-core
 * operand form, or the hidden activations [T x d_ff] f32 on the CUDA-core
 * path), rounded up to 256.  The size depends on d_model (the split token
 * operand is T x d_model) and on the group and shape (which path runs), not
 * only on T and d_ff, so all four sizes are arguments.
 * Returns (size_t)-1 for shapes the call would refuse (checked first, for
 * any T) and 0 for T <= 0.
 */
size_t smoe_ffn_batch_workspace_bytes(int T, int d_model, int d_ff, int group);

/*
 * Token-batch fused FFN of one Q4 expert ("Token-Batch Fused FFN"): the
 * one-token FFN above applied to every row of X:
 *
 *   H[t][i] = SiLU(gate . X[t])[i] * (up . X[t])[i]
 *   Y[t][j] = (down . H[t])[j]
 *
 * gate/up: packed Q4 [d_ff x d_model] with f32 scales [d_ff x d_model/group];
 * down: packed Q4 [d_model x d_ff] with f32 scales [d_model x d_ff/group].
 * X: f32 [T x d_model] row-major; Y: f32 [T x d_model], written.
 * workspace: device memory of at least
 * smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group) bytes, 16-byte
 * aligned, owned by the caller; its contents on entry do not matter and on
 * return are unspecified.  Two calls in flight at once need two workspaces.
 * The batch is not limited to the page's 64 tokens: any T >= 0 is accepted.
 * T = 1 runs on the decode kernels, 2 <= T <= 6 as one decode slot per token
 * (up to 8 where the tensor cores do not take the shape); larger T runs the
 * contraction on the tensor cores (codes as exact bf16 integers, X split
 * into two bf16 halves, f32 accumulation).
 */
int ffn_batch_q4(const uint8_t *gate_codes, const float *gate_scales,
                 const uint8_t *up_codes, const float *up_scales,
                 const uint8_t *down_codes, const float *down_scales,
                 const float *X, float *Y,
                 int T, int d_model, int d_ff, int group,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * The same token batch for one Q2 expert (the page names Q2 vaults as the
 * next format of this batched path): codes packed four per byte as in
 * smoe_gate_up_q2, Z = 1.5; d_model, d_ff and group multiples of 64 (the Q2
 * layout contract).  Same arguments, workspace size
 * (smoe_ffn_batch_workspace_bytes), checks and results as ffn_batch_q4;
 * the same paths by T, the tensor cores with A = (code - 1.5)/4 exact in
 * bf16.
 */
int ffn_batch_q2(const uint8_t *gate_codes, const float *gate_scales,
                 const uint8_t *up_codes, const float *up_scales,
                 const uint8_t *down_codes, const float *down_scales,
                 const float *X, float *Y,
                 int T, int d_model, int d_ff, int group,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Token batches of several experts in one submission ("Token-Batch Fused
 * FFN", applied per claimed expert: every expert with routed tokens gets its
 * own token matrix): for e in [0, n_experts), expert e's FFN over its T[e]
 * tokens,
 *
 *   Y[e][t] = down_e . (SiLU(gate_e . X[e][t]) * (up_e . X[e][t])),  t < T[e].
 *
 * gate_codes .. down_scales: host arrays of n_experts device pointers, each
 * expert laid out as for ffn_batch_q4 / ffn_batch_q2; X, Y: host arrays of
 * device pointers to f32 [T[e] x d_model]; T: host array of token counts
 * (>= 0; an expert with T[e] == 0 is skipped and may hold null pointers).
 * One shape (d_model, d_ff, group) for all experts.  When d_model, d_ff and
 * group are multiples of 64 every expert's token tiles share one grid per
 * 32 experts (three launches), so many small batches pay one launch ramp;
 * other shapes run expert after expert.  workspace: at least
 * smoe_experts_ffn_batch_workspace_bytes(n_experts, T, d_model, d_ff, group)
 * bytes, 16-byte aligned, caller-owned, contents unspecified on return.
 * No output may overlap any input, the workspace or another output.
 */
size_t smoe_experts_ffn_batch_workspace_bytes(int n_experts, const int *T,
                                              int d_model, int d_ff, int group);
int smoe_experts_ffn_batch_q4(int n_experts, const uint8_t *const *gate_codes,
                              const float *const *gate_scales,
                              const uint8_t *const *up_codes,
                              const float *const *up_scales,
                              const uint8_t *const *down_codes,
                              const float *const *down_scales,
                              const float *const *X, float *const *Y,
                              const int *T, int d_model, int d_ff, int group,
                              void *workspace, size_t workspace_bytes,
                              void *stream);
int smoe_experts_ffn_batch_q2(int n_experts, const uint8_t *const *gate_codes,
                              const float *const *gate_scales,
                              const uint8_t *const *up_codes,
                              const float *const *up_scales,
                              const uint8_t *const *down_codes,
                              const float *const *down_scales,
                              const float *const *X, float *const *Y,
                              const int *T, int d_model, int d_ff, int group,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/* Limits of smoe_route_topk_bf16. */
#define SMOE_MAX_TOP_K 64
#define SMOE_MAX_ROUTE_EXPERTS 8192

/*
 * Router of one token: logits of a bf16 gate matrix and the top-k experts
 * with their weights.  The page runs this "exact-routing gate matvec"
 * (n_experts x d_model) on the host and leaves selection and weighting
 * open; the reading implemented here:
 *
 *   logits[e] = sum_k bf16(gate_w[e][k]) * x[k]          (as matvec_bf16)
 *   top_idx   = the k largest logits in descending order, ties to the lower
 *               expert index, NaN below every number
 *   top_w[r]  = exp(logits[top_idx[r]] - logits[top_idx[0]])
 *               / sum over r' < k of exp(logits[top_idx[r']] - logits[top_idx[0]])
 *
 * gate_w: bf16 [n_experts x d_model]; x: f32 [d_model]; logits: f32
 * [n_experts], top_idx: int32 [k], top_w: f32 [k], all device memory
 * written by the call (16-byte aligned inputs; outputs 4-byte aligned).
 * 1 <= k <= min(n_experts, SMOE_MAX_TOP_K), n_experts <=
 * SMOE_MAX_ROUTE_EXPERTS, d_model a multiple of 8 and at most SMOE_MAX_COLS.
 * Outputs may not overlap inputs or each other.  Two launches (the matvec,
 * then one CTA for the selection).
 */
int smoe_route_topk_bf16(const uint16_t *gate_w, const float *x, int n_experts,
                         int d_model, int k, float *logits, int *top_idx,
                         float *top_w, void *stream);

/*
 * Weighted combine of a token's k expert outputs (the reading above):
 *
 *   out[j] = sum over r < k, in order, of top_w[r] * expert_out[r][j]
 *
 * expert_out: f32 [k x d_model] (row r the output of the r-th selected
 * expert, e.g. rows of smoe_experts_ffn_q4's out in selection order); top_w:
 * f32 [k] on the device; out: f32 [d_model], written.  k >= 0 (k == 0
 * writes zeros); out may not overlap the inputs.
 */
int smoe_combine(int k, const float *expert_out, const float *top_w,
                 float *out, int d_model, void *stream);

/* Most selected experts one routed call serves. */
#define SMOE_MAX_ROUTED_SLOTS 64

/*
 * Bytes of device workspace smoe_experts_ffn_routed_q4/q2 need: the hidden
 * activations [k x d_ff] f32, rounded up to 256.  (size_t)-1 for k < 0,
 * k > SMOE_MAX_ROUTED_SLOTS or d_ff < 0.
 */
size_t smoe_experts_ffn_routed_workspace_bytes(int k, int d_ff);

/*
 * Routed expert FFN of one token with the selection on the device
 * ("Grouped Expert Dispatch": all ready experts in one submission, with the
 * "exact-routing gate matvec" feeding it): for r < k, with e = top_idx[r],
 *
 *   out[r] = down_e . (SiLU(gate_e . x) * (up_e . x))
 *
 * so that smoe_route_topk_bf16 -> smoe_experts_ffn_routed_q4 -> smoe_combine
 * is a whole MoE layer with no host round trip (it can be captured in one
 * CUDA graph).  The expert indices are read on the device, after the
 * previous kernel in the stream has completed (top_idx is typically written
 * by smoe_route_topk_bf16 just before).
 *
 * gate_codes .. down_scales: DEVICE arrays of n_experts device pointers (a
 *   table built once when the weights are loaded, 8-byte aligned); entry e
 *   points to expert e's tensors with the layouts of smoe_gate_up_q4 and
 *   smoe_down_q4, 16-byte aligned.  The host cannot read these tables: an
 *   index outside [0, n_experts) or a table entry that is null or not
 *   16-byte aligned is caught on the device, before any load through it;
 *   that slot's outputs are then NaN and smoe_last_device_status returns
 *   SMOE_ERR_ROUTE.  Entries must otherwise point to tensors of the stated
 *   sizes.
 * top_idx: int32 [k] on the device.  x: f32 [d_model].  out: f32
 *   [k x d_model], written (row r for the r-th selected expert).
 * workspace: at least smoe_experts_ffn_routed_workspace_bytes(k, d_ff)
 *   bytes, 16-byte aligned (hidden activations; contents unspecified on
 *   return).  Calls in flight at once need separate workspaces.
 * 0 <= k <= SMOE_MAX_ROUTED_SLOTS; layout contract of the Q4 (Q2) calls;
 * d_model and d_ff multiples of 256 (Q4) or 512 (Q2), at most 8192 (rows of
 * whole multiples of 8 chunks of 16 bytes, which the bulk-copy decode
 * kernels take; e.g. d_model 4096, d_ff 1536), else SMOE_ERR_SHAPE.
 * k == 0 or d_model == 0: no-op; d_ff == 0: out is zeroed.
 * Two launches (gate/up of the k slots, then their down projections).
 */
int smoe_experts_ffn_routed_q4(int n_experts, int k,
                               const uint8_t *const *gate_codes,
                               const float *const *gate_scales,
                               const uint8_t *const *up_codes,
                               const float *const *up_scales,
                               const uint8_t *const *down_codes,
                               const float *const *down_scales,
                               const int *top_idx, const float *x, float *out,
                               int d_model, int d_ff, int group,
                               void *workspace, size_t workspace_bytes,
                               void *stream);

/* The same for Q2 weights (Z = 1.5, layout contract of smoe_gate_up_q2). */
int smoe_experts_ffn_routed_q2(int n_experts, int k,
                               const uint8_t *const *gate_codes,
                               const float *const *gate_scales,
                               const uint8_t *const *up_codes,
                               const float *const *up_scales,
                               const uint8_t *const *down_codes,
                               const float *const *down_scales,
                               const int *top_idx, const float *x, float *out,
                               int d_model, int d_ff, int group,
                               void *workspace, size_t workspace_bytes,
                               void *stream);

/* Size of the device array ffn_batch_q4_noalloc uses as its workspace. */
#define SMOE_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * ffn_batch_q4 for callers that must not allocate device memory: a host
 * program that has already divided all device memory among its own pools, a
 * plugin loaded into such a program, or a latency-critical caller for which
 * cudaMalloc's implicit device-wide synchronisation is not acceptable.  The
 * S-MoE page has no counterpart to this entry point; it exists only for such
 * callers.
 *
 * Same arguments, results and checks as ffn_batch_q4, without `workspace`:
 * the workspace is a file-scope device array of SMOE_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until
 * the process exits.  Shapes are checked first, as in ffn_batch_q4 (T == 0
 * with an invalid shape is refused too).  Calls whose workspace need,
 * smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group), exceeds that size
 * are refused with SMOE_ERR_SHAPE before anything is launched (at
 * d_model = 4096, d_ff = 1536 every T up to 256 fits; for T >= 2 the
 * workspace holds the split token operands of the tensor-core path and the
 * hidden activations in the down projection's operand form).
 * The function calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress while that device is current; make that first call
 * before any stream capture on the device.  All calls share the one array,
 * and it keeps the last call's contents: calls that overlap on the GPU (on
 * different streams, or from different host threads without ordering) race
 * on it and must be serialised by the caller.
 */
int ffn_batch_q4_noalloc(const uint8_t *gate_codes, const float *gate_scales,
                         const uint8_t *up_codes, const float *up_scales,
                         const uint8_t *down_codes, const float *down_scales,
                         const float *X, float *Y,
                         int T, int d_model, int d_ff, int group, void *stream);

/*
 * Reads and clears the library's device status word for the current device
 * after synchronising `stream`.  Kernels that wait on the device (bounded
 * mbarrier waits of the tensor-core batch path) set it when a wait gives up
 * instead of hanging; such a kernel skips its remaining work and exits.
 * Returns SMOE_OK, SMOE_ERR_TIMEOUT, SMOE_ERR_ROUTE (a routed call met an
 * invalid expert index or table entry), or SMOE_ERR_LAUNCH if the stream or
 * the status word cannot be read.
 */
int smoe_last_device_status(void *stream);

/*
 * dst[0 .. bytes) = src[0 .. bytes), copied by the SMs (not a copy engine)
 * so that a step's input and output transfers run in the same chain of
 * kernels as its compute (programmatic dependent launch on both sides; the
 * copy waits for the kernel before it, since that kernel may still read
 * dst).  Each buffer may be device memory, managed memory or pinned host
 * memory (cudaHostAlloc / cudaHostRegister / a pinned tensor), which the
 * SMs read and write over the host link; the caller owns both.  Both
 * pointers and `bytes` must be multiples of 16.  Asynchronous on `stream`.
 * Returns SMOE_OK (bytes == 0 is a no-op), SMOE_ERR_NULL, SMOE_ERR_ALIGN,
 * SMOE_ERR_ALIAS when the ranges overlap, SMOE_ERR_MEMORY when a buffer is
 * pageable host memory or unknown to CUDA, SMOE_ERR_LAUNCH.
 */
int smoe_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * Diagnostic of the device-side failure detection: launches one warp whose
 * bounded wait can never succeed -- kind 0: an mbarrier that expects two
 * arrivals and gets one; kind 1: a device counter that nothing increments --
 * with the limit the kernels use (about two seconds of SM clock).  The wait
 * gives up, records a timeout in the status word and the warp returns with
 * nothing in flight, so the context stays usable; the next
 * smoe_last_device_status(stream) returns SMOE_ERR_TIMEOUT.  Asynchronous:
 * returns SMOE_OK once launched, SMOE_ERR_SHAPE for another kind, and
 * SMOE_ERR_LAUNCH if CUDA refuses the launch.
 */
int smoe_selftest_bounded_wait(int kind, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SMOE_H */
