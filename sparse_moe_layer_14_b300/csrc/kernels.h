// Host-side launchers of the Beam MoE kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace beammoe {

struct ScheduleArgs;  // schedule.cuh

// ---- router (router.cu) ----
// FP32 SIMT router for small batches: logits[T][E] = x . W_r (a fixed-order
// split over the hidden dimension inside thread-block clusters), then sigmoid
// scores, group-limited top-k (on scores + sel_bias when sel_bias [E] is
// given) and normalised weights (unbiased scores). With
// router_simt_selects(T) the logits kernel selects too, counting finished CTAs
// in `ticket` (kRouteTickets ints, zero before the first call; the kernel
// returns them to zero); otherwise a selection kernel follows. `scratch` holds
// router_simt_scratch_bytes(d, E) bytes (a W_r copy with rows padded to a
// multiple of 4 experts when E is not one).
constexpr int kRouteTickets = 192;
bool router_simt_selects(int T);
size_t router_simt_scratch_bytes(int d, int E);
cudaError_t launch_router_simt(const uint16_t* x, const float* w_r, void* scratch, float* logits, int32_t* ticket,
                               int T, int d, int E, int n_groups, int topk_groups, int top_k, float routed_scale,
                               const float* sel_bias, int32_t* topk_idx, float* topk_w, int32_t* status,
                               int32_t* timeout_where, long long wait_spins, int num_sms, cudaStream_t stream);

// Tensor-core router for large batches (T >= kRouterTcMinTokens): W_r split
// into three bf16 terms, partial logits on the tensor cores, a warp-per-token
// selection that flags tokens with a narrow decision margin, and an fp32
// FFMA recompute of all logits of the flagged tokens.
// `scratch` holds router_tc_scratch_bytes(T, d, E) bytes.
constexpr int kRouterTcMinTokens = 1024;
constexpr int kRouterFlagSplits = 16;  // hidden-dimension parts of the fp32 recompute: [16][flagged][E] in `part`
int router_epad(int E);
bool router_uses_tensor_cores(int T, int E, int d);
size_t router_tc_scratch_bytes(int T, int d, int E);
int router_tc_splits(int T, int d, int num_sms);  // partial-logit buffers: [splits][T][E] fp32 in `part`
// `hdr_ticket` (8 ints, zero before the first call; the kernels return them
// to zero) and `timeout_where` live in the workspace header; `wait_spins`
// bounds the router's pipeline waits (see moe_set_wait_bound).
cudaError_t launch_router_tc(const uint16_t* x, const float* w_r, void* scratch, float* part, int32_t* flagged_count,
                             int32_t* hdr_ticket, int T, int d, int E, int n_groups, int topk_groups, int top_k,
                             float routed_scale, const float* sel_bias, int32_t* topk_idx, float* topk_w,
                             int32_t* status, int32_t* timeout_where, long long wait_spins, int num_sms,
                             cudaStream_t stream);

// ---- permutation (permute.cu) ----
int bitmap_words(int T);
size_t bitmap_bytes(int T, int E);
// Small batches (the bitmap fits in one CTA's shared memory) take one plan kernel for the
// bitmap, prefixes, counts and offsets; it needs no cleared bitmap, and given `sched` it also
// builds the expert GEMMs' work items.
bool permute_uses_plan_kernel(int T, int E);
// bitmap_zeroed: the caller has already cleared the bitmap on `stream` (otherwise, unless the
// plan kernel runs, a memset is enqueued first).
cudaError_t launch_permute(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int top_k,
                           uint32_t* bitmap, int32_t* word_prefix, int32_t* counts, int32_t* offsets,
                           int32_t* row_token, int32_t* inv_row, uint16_t* x_perm, int32_t* status,
                           cudaStream_t stream, bool bitmap_zeroed = false, const ScheduleArgs* sched = nullptr);

// ---- expert FFN (expert_gemm.cu) ----
struct ExpertPlan {
  int n_max;        // max tokens per work item (multiple of 16, <= 256)
  int max_tiles;    // upper bound of (expert, token tile) pairs
  int wtiles1;      // 128-row weight tiles per expert in GEMM1 (ceil(inter/128))
  int wtiles2;      // 256-row weight tiles per expert in GEMM2 (ceil(d/256))
};
// decoded: NVFP4 or FP8 weights (decoded into tensor memory; token tile <= 192)
ExpertPlan plan_experts(int T, int d, int E, int top_k, int inter, bool decoded);

struct ExpertBuffers {
  const uint16_t* x_perm;  // [R][d]
  const int32_t* offsets;  // [E+1]
  uint16_t* h;             // [R][inter]
  uint16_t* y;             // [R][d] bf16 output (dense MLP), or null
  float* y_f32;            // [R][d] fp32 output (the experts), or null
  int4* table;             // work schedule [E] (schedule.cuh)
  int32_t* tile_expert;    // [max_tiles]
  int32_t* n_items;        // [2]
  int32_t* status;
  int32_t* timeout_where;
};

struct ExpertWeightsDev {
  int wfmt;
  const void *gate, *up, *down;
  const void *gate_sf, *up_sf, *down_sf;  // e4m3 bytes (NVFP4) or fp32 (FP8)
  const float *gate_ts, *up_ts, *down_ts;
};

// items_ready: the work items were already built on the stream (by the permutation's plan
// kernel, from the same plan and buffers); otherwise a schedule kernel builds them first.
cudaError_t launch_expert_ffn(const ExpertPlan& plan, const ExpertBuffers& buf, const ExpertWeightsDev& w, int T,
                              int d, int E, int top_k, int inter, int num_sms, long long wait_spins,
                              cudaStream_t stream, int* cu_error, cudaEvent_t after_gemm1 = nullptr,
                              bool items_ready = false);
ScheduleArgs schedule_args(const ExpertPlan& plan, const ExpertBuffers& buf, int R);

// ---- pre-norm (norm.cu) ----
// x [T][d] = bf16(RMSNorm(h) * gain), FP32; d a multiple of 64; x must not overlap h.
cudaError_t launch_pre_norm(const uint16_t* h, const uint16_t* gain, float eps, uint16_t* x, int T, int d,
                            cudaStream_t stream);

// ---- combine (combine.cu) ----
// combine + post-norm (RMSNorm, gain [d]) + depth-scaled residual update of
// resid [T][d] in place at step `step` (>= 1); d <= 8192 (one cluster of
// <= 8 blocks per row).
cudaError_t launch_combine_residual(const float* y_perm, const int32_t* inv_row, const float* topk_w,
                                    const uint16_t* gain, float eps, int step, uint16_t* resid, int T, int d,
                                    int top_k, int32_t* status, cudaStream_t stream);
cudaError_t launch_combine(const float* y_perm, const int32_t* inv_row, const float* topk_w, uint16_t* out,
                           int T, int d, int top_k, int32_t* status, cudaStream_t stream);

}  // namespace beammoe
