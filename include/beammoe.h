/*
 * beammoe.h -- C ABI of the Beam MoE block forward pass on one NVIDIA B300.
 *
 * The block (Reflection "Beam 1.0" release article, section "Mixture of
 * Experts: 256 experts, 8 routed per token"; FP32 placement from section
 * "Residual stream", last paragraph):
 *   1. route    : logits = x . W_r in FP32, s = sigmoid(logits); experts split
 *                 into n_groups groups; group score = sum of the group's two
 *                 best s; keep the topk_groups best groups; choose the top_k
 *                 best experts inside them; weight = routed_scale * s / sum(s).
 *   2. permute  : group the (token, slot) pairs by expert.
 *   3. expert   : per chosen expert, SwiGLU MLP y = (silu(x Wg) * (x Wu)) Wd,
 *                 with the product silu(g) * u taken in FP32.
 *   4. combine  : out[t] = sum_k weight[t,k] * y[t,k]. No shared expert.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers, row-major, 16-byte aligned, and
 *    owned by the caller. The library never allocates or frees memory.
 *  - Every call is asynchronous: it validates its arguments on the host, then
 *    enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns. Invalid arguments return an error code before any
 *    launch. Launch failures return MOE_ERR_CUDA.
 *  - Errors found on the device (an expert id out of range, a row index out
 *    of range, a bounded wait that expired, a zero score sum) never trap:
 *    the kernel latches a code in the workspace header and skips the bad
 *    element. Read it with moe_get_device_status().
 *  - bf16 tensors are passed as their 16-bit patterns (moe_bf16_t).
 *  - Expert weights are stored K-contiguous: gate and up are [E][inter][d]
 *    (row i of expert e is column i of that expert's W_gate / W_up), down is
 *    [E][d][inter] (row n is column n of W_down). The router weight W_r is
 *    [d][E] fp32, logits = x . W_r.
 *  - NVFP4 weights: packed e2m1 codes [E][N][K/2] (low nibble = even k,
 *    nibble bit 3 = sign), e4m3 block scales [E][N][K/16] (one per 16
 *    consecutive k), one fp32 tensor scale per expert and matrix; the weight
 *    is e2m1 * e4m3 * tensor_scale.
 *  - FP8 weights (DeepSeek-V3's block-scaled layout): e4m3 codes [E][N][K]
 *    (one byte per weight), fp32 scales [E][N/128][K/128] (one per 128 x 128
 *    block of each expert's matrix); the weight is e4m3 * block scale. N and K
 *    (d and inter) must be multiples of 128.
 *  - Routing order: slots of a token are in descending score order, ties to
 *    the lower expert index; within an expert, permuted rows are ordered by
 *    ascending token.
 *  - Calls that share a workspace must not overlap in time (use one stream).
 */
#ifndef BEAMMOE_H
#define BEAMMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t; /* bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent dims */
  MOE_ERR_UNSUPPORTED = 2,   /* dims outside what the kernels implement (see moe_dims_t) */
  MOE_ERR_WORKSPACE = 3,     /* workspace null, misaligned or smaller than moe_workspace_bytes() */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_DEVICE_STATUS = 5, /* reserved for callers that fold the device code into one status */
  MOE_ERR_DEVICE_TIMEOUT = 6, /* device code: a bounded wait inside a kernel expired */
  MOE_ERR_SCRATCH_LIMIT = 7   /* moe_permute_noalloc: sizes beyond its fixed device scratch */
} moe_status_t;

/* Codes latched in the workspace header by kernels (read by moe_get_device_status). */
typedef enum {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_EXPERT = 1,  /* a routing index outside [0, E): the slot is skipped */
  MOE_DEV_BAD_ROW = 2,     /* a permuted-row index outside [0, T*top_k): skipped */
  MOE_DEV_DUP_EXPERT = 3,  /* a token names one expert in two slots: the slots share one row */
  MOE_DEV_TIMEOUT = 6,     /* a pipeline wait exceeded its bound; the kernel returned early */
  MOE_DEV_ZERO_SUM = 7,    /* a token's chosen scores summed to 0: its weights are set to 0 */
  MOE_DEV_CHECK = 8        /* debug build only: an index failed its bounds check; the access was skipped */
} moe_device_code_t;

typedef enum { MOE_W_BF16 = 0, MOE_W_NVFP4 = 1, MOE_W_FP8 = 2 } moe_wfmt_t;

/* Block shape. Beam: d=5120, E=256, n_groups=8, topk_groups=4, top_k=8,
 * inter=2560, routed_scale=2.5 (release article, "Mixture of Experts").
 * Supported: T >= 0 (T == 0 is a no-op), d and inter multiples of 64 and at
 * most 16384, 1 <= E <= 256, n_groups divides E and n_groups <= 32,
 * 1 <= topk_groups <= n_groups, 1 <= top_k <= min(32, topk_groups*E/n_groups),
 * T <= 4194304. Calls that run the expert GEMMs return MOE_ERR_UNSUPPORTED
 * unless d and inter are multiples of 256 for MOE_W_NVFP4 and of 128 for
 * MOE_W_FP8. */
typedef struct {
  int32_t T;
  int32_t d;
  int32_t E;
  int32_t n_groups;
  int32_t topk_groups;
  int32_t top_k;
  int32_t inter;
  float routed_scale;
  int32_t wfmt; /* moe_wfmt_t */
} moe_dims_t;

/* Expert weights (device pointers, 16-byte aligned). For MOE_W_BF16 only
 * gate/up/down are read (bf16, layouts above). For MOE_W_NVFP4 gate/up/down
 * are the packed e2m1 codes and the *_sf (e4m3 bytes) and *_ts fields are
 * required. For MOE_W_FP8 gate/up/down are the e4m3 codes and *_sf point at
 * the fp32 block scales (4-byte aligned); *_ts are ignored. The caller owns
 * all of them; calls only read them. */
typedef struct {
  const void* gate;
  const void* up;
  const void* down;
  const void* gate_sf;
  const void* up_sf;
  const void* down_sf;
  const float* gate_ts;
  const float* up_ts;
  const float* down_ts;
} moe_expert_weights_t;

/* Bytes of device workspace every call below needs for these dims (one size
 * for all calls). The workspace is caller-owned and may be reused across
 * calls on one stream. It must be 256-byte aligned. */
size_t moe_workspace_bytes(const moe_dims_t* dims);

/* Zero the workspace header (the device status word). Call once after
 * allocating a workspace; asynchronous on `stream`. */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Step 1, router (article section "Mixture of Experts"; FP32 per section
 * "Residual stream"). x [T][d] bf16, w_r [d][E] fp32 ->
 * topk_idx [T][top_k] int32 (expert ids, descending score, ties to lower id),
 * topk_w [T][top_k] fp32 (routed_scale * s / sum of the token's chosen s).
 * Below 1,024 tokens the logits are FP32 FMA sums in a fixed order; from
 * 1,024 tokens they come from the tensor cores (an exact three-way bf16 split
 * of w_r), and every token whose decision margins lie within the bound of
 * that path's accumulation error is routed again from FP32 FMA logits. The
 * result is deterministic for given inputs. */
moe_status_t moe_route(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r,
                       int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* Step 2, permutation: group the T*top_k (token, slot) pairs by expert.
 * counts [E]: tokens routed to each expert; offsets [E+1]: exclusive prefix
 * sum of counts (offsets[E] = T*top_k); row_token [T*top_k]: token of each
 * permuted row (rows of expert e are offsets[e]..offsets[e+1]-1, tokens
 * ascending); inv_row [T*top_k]: permuted row of token t's slot k at
 * t*top_k+k; x_perm [T*top_k][d] bf16: x[row_token[r]] for every row r.
 * Indices outside [0, E) latch MOE_DEV_BAD_EXPERT and are dropped. A token
 * that names the same expert in two slots (the router never does) latches
 * MOE_DEV_DUP_EXPERT: both slots get one shared row (inv_row equal), counts
 * count the token once, so offsets[E] = T*top_k minus the repeats; a combine
 * over inv_row still adds that row once per slot. */
moe_status_t moe_permute(const moe_dims_t* dims, const moe_bf16_t* x, const int32_t* topk_idx,
                         int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* inv_row,
                         moe_bf16_t* x_perm, void* ws, size_t ws_bytes, void* stream);

/* Step 3, experts (article section "Mixture of Experts": SwiGLU experts,
 * intermediate size 2,560; product in FP32 per section "Residual stream").
 * For every expert e and permuted row r in [offsets[e], offsets[e+1]):
 *   h = bf16( silu(x_perm[r] . Wg_e) * (x_perm[r] . Wu_e) )   (FP32 math)
 *   y_perm[r] = h . Wd_e                                       (FP32 accumulate)
 * x_perm [T*top_k][d] bf16, offsets [E+1] int32 (non-decreasing, offsets[0]=0,
 * offsets[E] <= T*top_k), y_perm [T*top_k][d] fp32 (the expert output kept in
 * FP32: the block output is its only rounding after h). The GEMMs run on tcgen05
 * tensor cores with bf16 operands (NVFP4 weights are decoded to exact bf16
 * values on chip, the tensor scale applied to the FP32 accumulator; FP8
 * weights are decoded on chip as bf16(e4m3 * block scale), the product in
 * FP32, rounded once). */
moe_status_t moe_expert_ffn(const moe_dims_t* dims, const moe_bf16_t* x_perm,
                            const int32_t* offsets, const moe_expert_weights_t* weights,
                            float* y_perm, void* ws, size_t ws_bytes, void* stream);

/* Step 4, combine (article section "Mixture of Experts": weighted by the
 * normalised, 2.5-scaled router weights; no shared expert):
 * out[t] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*top_k+k]] ), FP32 sum
 * in slot order. y_perm [T*top_k][d] fp32 (16-byte aligned), out [T][d] bf16. Rows outside [0, T*top_k) latch
 * MOE_DEV_BAD_ROW and are skipped; needs no workspace except for that code. */
moe_status_t moe_combine(const moe_dims_t* dims, const float* y_perm, const int32_t* inv_row,
                         const float* topk_w, moe_bf16_t* out, void* ws, size_t ws_bytes,
                         void* stream);

/* The whole block: route -> permute -> experts -> combine, all on `stream`,
 * with no host synchronisation. x [T][d] bf16, w_r [d][E] fp32, out [T][d]
 * bf16. topk_idx [T][top_k] and counts [E] are optional outputs (NULL to
 * skip). Intermediates live in the workspace. */
moe_status_t moe_forward(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r,
                         const moe_expert_weights_t* weights, moe_bf16_t* out, int32_t* topk_idx,
                         int32_t* counts, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free permutation. The block's description has no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- code running while
 * a CUDA graph is captured, serving loops that must never call cudaMalloc, or
 * plugins whose host framework owns all device memory. It computes exactly
 * what moe_permute computes, with the same arguments except the workspace:
 * its scratch (a token x expert bitmap and per-word prefix counts, plus a
 * status word) lives in one fixed device array of about 1 MiB inside the
 * library, which every GPU that loads the library keeps until the process
 * exits. Nothing is allocated and no allocating routine is called.
 * Limits: T <= 16384 and E <= 256; larger sizes return MOE_ERR_SCRATCH_LIMIT
 * before any work. The first call on each device looks up the array's device
 * address (one-time set-up), so make that first call before any stream
 * capture. All calls share the array and it keeps the last call's contents:
 * every call clears its status word and bitmap first, and calls that overlap
 * on the GPU (other streams, other host threads) race on it -- issue them on
 * one stream. device_status (device int32, nullable) receives this call's
 * moe_device_code_t (MOE_DEV_BAD_EXPERT if an index was out of range,
 * MOE_DEV_DUP_EXPERT if a token repeated an expert; MOE_DEV_OK when T == 0). */
moe_status_t moe_permute_noalloc(const moe_dims_t* dims, const moe_bf16_t* x, const int32_t* topk_idx,
                                 int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* inv_row,
                                 moe_bf16_t* x_perm, int32_t* device_status, void* stream);

/* moe_route and moe_forward with a per-expert selection bias (nullable
 * sel_bias [E] fp32, 4-byte aligned): the auxiliary-loss-free balancing bias
 * of DeepSeek-V3's router, which the article's router follows (release
 * article, section "Mixture of Experts"; the pre-training notes mention
 * expert-bias updates). Group scores (top-2 sums) and the expert choice use
 * s + sel_bias (FP32 add); the combine weights use the unbiased s:
 * w = routed_scale * s / sum of the chosen s. Slot order is descending
 * s + sel_bias. sel_bias = NULL is moe_route / moe_forward. */
moe_status_t moe_route_ex(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                          int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream);
moe_status_t moe_forward_ex(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                            const moe_expert_weights_t* weights, moe_bf16_t* out, int32_t* topk_idx,
                            int32_t* counts, void* ws, size_t ws_bytes, void* stream);

/* Combine fused with the sublayer's post-norm and the depth-scaled residual
 * addition (release article, section "Residual stream": every sublayer is
 * normalised before and after; at step k the stream keeps weight
 * sqrt((k-1)/k) and takes the sublayer output with weight 1/sqrt(k), the input
 * embedding counting as step 1; the norms are computed in FP32). For every
 * token t, with out[t] = sum_k topk_w[t][k] * y_perm[inv_row[t*top_k+k]] (FP32,
 * slot order):
 *   r = sqrt(mean_c(out[t][c]^2) + eps)
 *   resid[t][c] = bf16( sqrt((step-1)/step) * resid[t][c]
 *                       + (1/sqrt(step)) * out[t][c] / r * norm_gain[c] )
 * in place. resid [T][d] bf16 and norm_gain [d] bf16 (the post-norm's RMSNorm
 * weight) 16-byte aligned; step >= 1; eps >= 0 (the pages give none; 1e-6 is
 * usual); d <= 8192 (larger d returns MOE_ERR_UNSUPPORTED). moe_forward_residual
 * is moe_forward_ex with this as its
 * last stage instead of writing out. */
moe_status_t moe_combine_residual(const moe_dims_t* dims, const float* y_perm, const int32_t* inv_row,
                                  const float* topk_w, const moe_bf16_t* norm_gain, float eps, int32_t step,
                                  moe_bf16_t* resid, void* ws, size_t ws_bytes, void* stream);
moe_status_t moe_forward_residual(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r,
                                  const float* sel_bias, const moe_expert_weights_t* weights,
                                  const moe_bf16_t* norm_gain, float eps, int32_t step, moe_bf16_t* resid,
                                  int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes, void* stream);

/* Pre-norm of a sublayer input (release article, section "Residual stream":
 * every sublayer is normalised before and after, the norms in FP32). For every
 * token t:
 *   x[t][c] = bf16( h[t][c] * gain[c] / sqrt(mean_c(h[t][c]^2) + eps) )   (FP32)
 * h, x [T][d] and gain [d] bf16, 16-byte aligned; x must not overlap h;
 * eps >= 0. Uses dims->T and dims->d (a multiple of 64, at most 16384); the
 * other fields are ignored. One kernel, no workspace. */
moe_status_t moe_pre_norm(const moe_dims_t* dims, const moe_bf16_t* h, const moe_bf16_t* gain, float eps,
                          moe_bf16_t* x, void* stream);

/* The MoE sublayer as a decoder layer runs it (release article, section
 * "Residual stream"): x = the pre-norm of resid with pre_gain (as
 * moe_pre_norm, into the caller's x [T][d], which must not overlap resid);
 * the block forward on x with the optional selection bias (as moe_forward_ex);
 * then the post-norm with post_gain and the depth-scaled update of resid in
 * place at step `step` (as moe_forward_residual). One eps for both norms;
 * d <= 8192. All arguments are checked before the first launch. */
moe_status_t moe_sublayer(const moe_dims_t* dims, moe_bf16_t* resid, const moe_bf16_t* pre_gain,
                          const moe_bf16_t* post_gain, float eps, int32_t step, const float* w_r,
                          const float* sel_bias, const moe_expert_weights_t* weights, moe_bf16_t* x,
                          int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes, void* stream);

/* Dense SwiGLU MLP of the first decoder layers (release article, section
 * "Architecture": the first 3 of the 52 layers use a dense SwiGLU MLP instead
 * of the Mixture-of-Experts block). For every token t:
 *   h = bf16( silu(x[t] . Wg) * (x[t] . Wu) )   (FP32 math, as for the experts)
 *   out[t] = bf16( h . Wd )                       (FP32 accumulate)
 * on the expert GEMM kernels with a single expert and no routing. Uses
 * dims->T, d, inter and wfmt; E, n_groups, topk_groups, top_k and
 * routed_scale are ignored. `w` holds one MLP in the expert layouts with E = 1
 * (gate, up [inter][d], down [d][inter]; NVFP4 as for the experts). x [T][d]
 * and out [T][d] bf16, 16-byte aligned; d a multiple of 64 up to 16384, inter
 * a multiple of 64 up to 65536 (NVFP4: both multiples of 256; FP8: of 128). The workspace
 * (moe_dense_workspace_bytes bytes, 256-byte aligned, header zeroed by
 * moe_workspace_init) holds the work items and h [T][inter]. Host-side errors
 * return before any launch; device codes latch in the workspace header. */
size_t moe_dense_workspace_bytes(const moe_dims_t* dims);
moe_status_t moe_dense_mlp(const moe_dims_t* dims, const moe_bf16_t* x, const moe_expert_weights_t* w,
                           moe_bf16_t* out, void* ws, size_t ws_bytes, void* stream);

/* Read (and with clear != 0, reset) the device code latched in the workspace
 * header. Synchronises `stream`. *code receives a moe_device_code_t. */
moe_status_t moe_get_device_status(void* ws, void* stream, int32_t clear, int32_t* code);

/* Test hook: bound (in spin iterations) of every pipeline wait in the expert
 * GEMM kernels and in the tensor-core router (its logits kernel and the FP32
 * recompute of narrow-margin tokens) of later calls in this process; 0
 * restores the default. A
 * bound of 1 makes a wait give up almost at once, which exercises the
 * timeout path (MOE_DEV_TIMEOUT) without faulting or hanging the GPU. */
void moe_set_wait_bound(int64_t spins);

/* Optional instrumentation. With events != NULL (n >= 6 cudaEvent_t handles,
 * created by the caller), every later moe_forward call records events[0]
 * before its first launch and events[i] after stage i on its stream:
 * 1 router, 2 permutation, 3 work-item schedule + expert GEMM1 (SwiGLU),
 * 4 expert GEMM2, 5 combine. cudaEventElapsedTime between consecutive events
 * then gives each stage's device time (moe_dense_mlp records events[0] before
 * its first launch, events[3] after GEMM1 and events[4] after GEMM2;
 * moe_sublayer records events[0] after its pre-norm). NULL (or
 * n < 6) turns it off. The
 * setting is process-wide; do not change it while moe_forward calls run on
 * other host threads. */
moe_status_t moe_set_stage_events(void* const* events, int32_t n);

/* Static description of the library build, e.g. "beammoe sm_103a". */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BEAMMOE_H */
