// C ABI of the Beam MoE block (declared in include/beammoe.h): argument
// validation, the workspace layout, and the launch sequence of each step.
// No call allocates memory or synchronises the host except
// moe_get_device_status().
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"

using namespace beammoe;

namespace {

constexpr size_t kAlign = 256;
constexpr long long kDefaultSpins = 1ll << 40;  // pipeline waits are bounded by time by default
long long g_wait_spins = kDefaultSpins;
cudaEvent_t g_stage_events[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
bool g_stage_events_on = false;

cudaError_t mark(int i, cudaStream_t s) {
  return g_stage_events_on ? cudaEventRecord(g_stage_events[i], s) : cudaSuccess;
}

// NVTX range around the host-side enqueue of one stage (named as the stage events are), so a
// timeline tool shows which launches belong to which step of the block; a no-op without a tool.
struct NvtxStage {
  explicit NvtxStage(const char* name) { nvtxRangePushA(name); }
  ~NvtxStage() { nvtxRangePop(); }
  NvtxStage(const NvtxStage&) = delete;
  NvtxStage& operator=(const NvtxStage&) = delete;
};

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

enum Region {
  R_HDR, R_PART, R_WSPLIT, R_BITMAP, R_WPRE, R_COUNTS, R_OFFS, R_IDX, R_W, R_ROWTOK, R_INVROW,
  R_SCHED, R_TILEX, R_XPERM, R_H, R_Y, R_NUM
};

struct Layout {
  size_t off[R_NUM];
  size_t total;
};

// Upper bound of SMs used to size the router's split-K buffer (the split
// factor grows with the SM count, so this bounds every device).
constexpr int kMaxSmsForLayout = 1024;

Layout make_layout(const moe_dims_t& d) {
  const int64_t T = d.T, R = T * d.top_k;
  const int Tc = d.T > 0 ? d.T : 1;
  const bool tc = router_uses_tensor_cores(d.T, d.E, d.d);
  const int splits = tc ? std::max(kRouterFlagSplits, router_tc_splits(Tc, d.d, kMaxSmsForLayout)) : 1;
  const ExpertPlan pl = plan_experts(d.T, d.d, d.E, d.top_k, d.inter, d.wfmt != MOE_W_BF16);
  const int64_t nw = bitmap_words(d.T);
  size_t sz[R_NUM];
  sz[R_HDR] = sizeof(WsHeader);
  sz[R_PART] = sizeof(float) * static_cast<size_t>(splits) * T * d.E;
  sz[R_WSPLIT] = tc ? router_tc_scratch_bytes(d.T, d.d, d.E) : router_simt_scratch_bytes(d.d, d.E);
  sz[R_BITMAP] = sizeof(uint32_t) * static_cast<size_t>(d.E) * nw;
  sz[R_WPRE] = sizeof(int32_t) * static_cast<size_t>(d.E) * nw;
  sz[R_COUNTS] = sizeof(int32_t) * d.E;
  sz[R_OFFS] = sizeof(int32_t) * (d.E + 1);
  sz[R_IDX] = sizeof(int32_t) * R;
  sz[R_W] = sizeof(float) * R;
  sz[R_ROWTOK] = sizeof(int32_t) * R;
  sz[R_INVROW] = sizeof(int32_t) * R;
  sz[R_SCHED] = sizeof(int4) * d.E;
  sz[R_TILEX] = sizeof(int32_t) * static_cast<size_t>(pl.max_tiles);
  sz[R_XPERM] = sizeof(uint16_t) * R * d.d;
  sz[R_H] = sizeof(uint16_t) * R * d.inter;
  sz[R_Y] = sizeof(float) * R * d.d;
  Layout L;
  size_t o = 0;
  for (int i = 0; i < R_NUM; ++i) {
    L.off[i] = o;
    o = align_up(o + sz[i]);
  }
  L.total = o;
  return L;
}

template <typename P>
P* region(void* ws, const Layout& L, Region r) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + L.off[r]);
}

moe_status_t check_dims(const moe_dims_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->d <= 0 || d->E <= 0 || d->n_groups <= 0 || d->topk_groups <= 0 || d->top_k <= 0 ||
      d->inter <= 0 || !std::isfinite(d->routed_scale))
    return MOE_ERR_INVALID_ARG;
  if (d->E % d->n_groups != 0 || d->topk_groups > d->n_groups || d->top_k > d->topk_groups * (d->E / d->n_groups))
    return MOE_ERR_INVALID_ARG;
  if (d->wfmt != MOE_W_BF16 && d->wfmt != MOE_W_NVFP4 && d->wfmt != MOE_W_FP8) return MOE_ERR_INVALID_ARG;
  if (d->T > 4194304 || d->d % 64 || d->inter % 64 || d->d > 16384 || d->inter > 16384 || d->E > 256 ||
      d->n_groups > 32 || d->top_k > 32)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_ws(const moe_dims_t* d, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < make_layout(*d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t check_weights(const moe_dims_t* d, const moe_expert_weights_t* w) {
  if (!w || !aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down)) return MOE_ERR_INVALID_ARG;
  if (d->wfmt == MOE_W_NVFP4) {
    if (!aligned16(w->gate_sf) || !aligned16(w->up_sf) || !aligned16(w->down_sf) || !w->gate_ts || !w->up_ts ||
        !w->down_ts)
      return MOE_ERR_INVALID_ARG;
  }
  if (d->wfmt == MOE_W_FP8) {
    const auto aligned4 = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!aligned4(w->gate_sf) || !aligned4(w->up_sf) || !aligned4(w->down_sf)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int32_t* status_word(void* ws) { return ws ? &reinterpret_cast<WsHeader*>(ws)->status : nullptr; }

moe_status_t do_route(const moe_dims_t* d, const uint16_t* x, const float* w_r, const float* sel_bias, int32_t* idx,
                      float* w, void* ws, const Layout& L, cudaStream_t s) {
  if (router_uses_tensor_cores(d->T, d->E, d->d)) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    return cuda_status(launch_router_tc(x, w_r, region<uint8_t>(ws, L, R_WSPLIT), region<float>(ws, L, R_PART),
                                        &hdr->router_flagged, hdr->wn_ticket, d->T, d->d, d->E, d->n_groups,
                                        d->topk_groups, d->top_k, d->routed_scale, sel_bias, idx, w, &hdr->status,
                                        &hdr->timeout_where, g_wait_spins, num_sms(), s));
  }
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  return cuda_status(launch_router_simt(x, w_r, region<uint8_t>(ws, L, R_WSPLIT), region<float>(ws, L, R_PART),
                                        hdr->route_ticket, d->T, d->d, d->E, d->n_groups, d->topk_groups, d->top_k,
                                        d->routed_scale, sel_bias, idx, w, &hdr->status, &hdr->timeout_where,
                                        g_wait_spins, num_sms(), s));
}

moe_status_t do_permute(const moe_dims_t* d, const uint16_t* x, const int32_t* idx, int32_t* counts,
                        int32_t* offsets, int32_t* row_token, int32_t* inv_row, uint16_t* x_perm, void* ws,
                        const Layout& L, cudaStream_t s, bool bitmap_zeroed = false,
                        const ScheduleArgs* sched = nullptr) {
  cudaError_t e = launch_permute(x, idx, d->T, d->d, d->E, d->top_k, region<uint32_t>(ws, L, R_BITMAP),
                                 region<int32_t>(ws, L, R_WPRE), counts, offsets, row_token, inv_row, x_perm,
                                 status_word(ws), s, bitmap_zeroed, sched);
  return cuda_status(e);
}

ExpertWeightsDev weights_dev(int wfmt, const moe_expert_weights_t* w) {
  ExpertWeightsDev wd;
  wd.wfmt = wfmt;
  wd.gate = w->gate;
  wd.up = w->up;
  wd.down = w->down;
  wd.gate_sf = w->gate_sf;
  wd.up_sf = w->up_sf;
  wd.down_sf = w->down_sf;
  wd.gate_ts = w->gate_ts;
  wd.up_ts = w->up_ts;
  wd.down_ts = w->down_ts;
  return wd;
}

ExpertBuffers expert_buffers(const uint16_t* x_perm, const int32_t* offsets, float* y, void* ws, const Layout& L) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  ExpertBuffers b{};
  b.x_perm = x_perm;
  b.offsets = offsets;
  b.h = region<uint16_t>(ws, L, R_H);
  b.y = nullptr;
  b.y_f32 = y;
  b.table = region<int4>(ws, L, R_SCHED);
  b.tile_expert = region<int32_t>(ws, L, R_TILEX);
  b.n_items = hdr->n_items;
  b.status = &hdr->status;
  b.timeout_where = &hdr->timeout_where;
  return b;
}

moe_status_t do_ffn(const moe_dims_t* d, const uint16_t* x_perm, const int32_t* offsets,
                    const moe_expert_weights_t* w, float* y, void* ws, const Layout& L, cudaStream_t s,
                    cudaEvent_t after_gemm1 = nullptr, bool items_ready = false) {
  const ExpertPlan pl = plan_experts(d->T, d->d, d->E, d->top_k, d->inter, d->wfmt != MOE_W_BF16);
  const ExpertBuffers b = expert_buffers(x_perm, offsets, y, ws, L);
  const ExpertWeightsDev wd = weights_dev(d->wfmt, w);
  int cu_err = 0;
  const cudaError_t e = launch_expert_ffn(pl, b, wd, d->T, d->d, d->E, d->top_k, d->inter, num_sms(), g_wait_spins,
                                          s, &cu_err, after_gemm1, items_ready);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_dims_t* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return make_layout(*dims).total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(WsHeader) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(WsHeader), static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_route_ex(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                          int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(w_r) || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes)) != MOE_OK) return st;
  return do_route(dims, x, w_r, sel_bias, topk_idx, topk_w, ws, make_layout(*dims),
                  static_cast<cudaStream_t>(stream));
}

moe_status_t moe_route(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, int32_t* topk_idx,
                       float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  return moe_route_ex(dims, x, w_r, nullptr, topk_idx, topk_w, ws, ws_bytes, stream);
}

moe_status_t moe_permute(const moe_dims_t* dims, const moe_bf16_t* x, const int32_t* topk_idx, int32_t* counts,
                         int32_t* offsets, int32_t* row_token, int32_t* inv_row, moe_bf16_t* x_perm, void* ws,
                         size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(x) || !topk_idx || !counts || !offsets || !row_token || !inv_row || !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes)) != MOE_OK) return st;
  return do_permute(dims, x, topk_idx, counts, offsets, row_token, inv_row, x_perm, ws, make_layout(*dims),
                    static_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn(const moe_dims_t* dims, const moe_bf16_t* x_perm, const int32_t* offsets,
                            const moe_expert_weights_t* weights, float* y_perm, void* ws, size_t ws_bytes,
                            void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(x_perm) || !offsets || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(dims, weights)) != MOE_OK) return st;
  if ((st = check_ws(dims, ws, ws_bytes)) != MOE_OK) return st;
  return do_ffn(dims, x_perm, offsets, weights, y_perm, ws, make_layout(*dims), static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_dims_t* dims, const float* y_perm, const int32_t* inv_row, const float* topk_w,
                         moe_bf16_t* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(y_perm) || !inv_row || !topk_w || !out || (reinterpret_cast<uintptr_t>(out) & 7u))
    return MOE_ERR_INVALID_ARG;
  if (ws && ws_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_combine(y_perm, inv_row, topk_w, out, dims->T, dims->d, dims->top_k, status_word(ws),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_forward(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r,
                         const moe_expert_weights_t* weights, moe_bf16_t* out, int32_t* topk_idx, int32_t* counts,
                         void* ws, size_t ws_bytes, void* stream) {
  return moe_forward_ex(dims, x, w_r, nullptr, weights, out, topk_idx, counts, ws, ws_bytes, stream);
}

// The fused forward; with res != nullptr the last stage is the combine fused
// with the post-norm and residual update of res->resid (no `out`).
struct ResidualArgs {
  const uint16_t* gain;
  float eps;
  int step;
  uint16_t* resid;
};

moe_status_t forward_impl(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                          const moe_expert_weights_t* weights, moe_bf16_t* out, const ResidualArgs* res,
                          int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
  if (!res && (!out || (reinterpret_cast<uintptr_t>(out) & 7u))) return MOE_ERR_INVALID_ARG;
  if (res && (!aligned16(res->resid) || !aligned16(res->gain) || res->step < 1 || !(res->eps >= 0.0f)))
    return MOE_ERR_INVALID_ARG;
  if (res && dims->d > 8192) return MOE_ERR_UNSUPPORTED;  // one cluster of <= 8 blocks per row
  if (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(dims, weights)) != MOE_OK) return st;
  if ((st = check_ws(dims, ws, ws_bytes)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = make_layout(*dims);
  int32_t* idx = topk_idx ? topk_idx : region<int32_t>(ws, L, R_IDX);
  float* w = region<float>(ws, L, R_W);
  int32_t* cnt = counts ? counts : region<int32_t>(ws, L, R_COUNTS);
  int32_t* offs = region<int32_t>(ws, L, R_OFFS);
  int32_t* row_token = region<int32_t>(ws, L, R_ROWTOK);
  int32_t* inv_row = region<int32_t>(ws, L, R_INVROW);
  uint16_t* x_perm = region<uint16_t>(ws, L, R_XPERM);
  float* y = region<float>(ws, L, R_Y);
  // The permutation also builds the expert GEMMs' work schedule (in its plan kernel for small
  // batches, in its offsets kernel otherwise). For larger batches its bitmap is cleared first,
  // so that no copy sits between the block's kernels (they launch back to back with
  // programmatic dependencies).
  const bool plan_kernel = permute_uses_plan_kernel(dims->T, dims->E);
  const ExpertPlan plan = plan_experts(dims->T, dims->d, dims->E, dims->top_k, dims->inter, dims->wfmt != MOE_W_BF16);
  const ScheduleArgs sched =
      schedule_args(plan, expert_buffers(x_perm, offs, y, ws, L), dims->T * dims->top_k);
  if (!plan_kernel &&
      cudaMemsetAsync(region<uint32_t>(ws, L, R_BITMAP), 0, bitmap_bytes(dims->T, dims->E), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (mark(0, s) != cudaSuccess) return MOE_ERR_CUDA;
  {
    NvtxStage r("moe router");
    if ((st = do_route(dims, x, w_r, sel_bias, idx, w, ws, L, s)) != MOE_OK) return st;
  }
  if (mark(1, s) != cudaSuccess) return MOE_ERR_CUDA;
  {
    NvtxStage r("moe permute");
    if ((st = do_permute(dims, x, idx, cnt, offs, row_token, inv_row, x_perm, ws, L, s, true,
                         &sched)) != MOE_OK)
      return st;
  }
  if (mark(2, s) != cudaSuccess) return MOE_ERR_CUDA;
  {
    NvtxStage r("moe expert GEMMs");
    if ((st = do_ffn(dims, x_perm, offs, weights, y, ws, L, s, g_stage_events_on ? g_stage_events[3] : nullptr,
                     true)) != MOE_OK)
      return st;
  }
  if (mark(4, s) != cudaSuccess) return MOE_ERR_CUDA;
  {
    NvtxStage r(res ? "moe combine + post-norm residual" : "moe combine");
    st = cuda_status(res ? launch_combine_residual(y, inv_row, w, res->gain, res->eps, res->step, res->resid, dims->T,
                                                   dims->d, dims->top_k, status_word(ws), s)
                         : launch_combine(y, inv_row, w, out, dims->T, dims->d, dims->top_k, status_word(ws), s));
  }
  if (st != MOE_OK) return st;
  return mark(5, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_forward_ex(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                            const moe_expert_weights_t* weights, moe_bf16_t* out, int32_t* topk_idx, int32_t* counts,
                            void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(dims, x, w_r, sel_bias, weights, out, nullptr, topk_idx, counts, ws, ws_bytes, stream);
}

moe_status_t moe_forward_residual(const moe_dims_t* dims, const moe_bf16_t* x, const float* w_r, const float* sel_bias,
                                  const moe_expert_weights_t* weights, const moe_bf16_t* norm_gain, float eps,
                                  int32_t step, moe_bf16_t* resid, int32_t* topk_idx, int32_t* counts, void* ws,
                                  size_t ws_bytes, void* stream) {
  const ResidualArgs res{norm_gain, eps, step, resid};
  return forward_impl(dims, x, w_r, sel_bias, weights, nullptr, &res, topk_idx, counts, ws, ws_bytes, stream);
}

moe_status_t moe_combine_residual(const moe_dims_t* dims, const float* y_perm, const int32_t* inv_row,
                                  const float* topk_w, const moe_bf16_t* norm_gain, float eps, int32_t step,
                                  moe_bf16_t* resid, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(y_perm) || !inv_row || !topk_w || !aligned16(norm_gain) || !aligned16(resid) || step < 1 ||
      !(eps >= 0.0f))
    return MOE_ERR_INVALID_ARG;
  if (dims->d > 8192) return MOE_ERR_UNSUPPORTED;
  if (ws && ws_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_combine_residual(y_perm, inv_row, topk_w, norm_gain, eps, step, resid, dims->T, dims->d,
                                             dims->top_k, status_word(ws), static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- pre-norm and the sublayer

namespace {

moe_status_t check_norm_args(const moe_dims_t* d, const void* h, const void* gain, float eps, const void* x) {
  if (!d || d->T < 0 || d->d <= 0) return MOE_ERR_INVALID_ARG;
  if (d->T > 4194304 || d->d % 64 || d->d > 16384) return MOE_ERR_UNSUPPORTED;
  if (d->T == 0) return MOE_OK;
  if (!aligned16(h) || !aligned16(gain) || !aligned16(x) || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  const uintptr_t hb = reinterpret_cast<uintptr_t>(h), xb = reinterpret_cast<uintptr_t>(x);
  const uintptr_t n = static_cast<uintptr_t>(d->T) * static_cast<uintptr_t>(d->d) * 2u;
  if (hb < xb + n && xb < hb + n) return MOE_ERR_INVALID_ARG;  // x overlaps h
  return MOE_OK;
}

}  // namespace

moe_status_t moe_pre_norm(const moe_dims_t* dims, const moe_bf16_t* h, const moe_bf16_t* gain, float eps,
                          moe_bf16_t* x, void* stream) {
  const moe_status_t st = check_norm_args(dims, h, gain, eps, x);
  if (st != MOE_OK || dims->T == 0) return st;
  return cuda_status(launch_pre_norm(h, gain, eps, x, dims->T, dims->d, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_sublayer(const moe_dims_t* dims, moe_bf16_t* resid, const moe_bf16_t* pre_gain,
                          const moe_bf16_t* post_gain, float eps, int32_t step, const float* w_r,
                          const float* sel_bias, const moe_expert_weights_t* weights, moe_bf16_t* x,
                          int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dims(dims);
  if (st != MOE_OK) return st;
  if ((st = check_norm_args(dims, resid, pre_gain, eps, x)) != MOE_OK || dims->T == 0) return st;
  // everything forward_impl checks, before the pre-norm is enqueued
  if (!aligned16(w_r) || !aligned16(post_gain) || step < 1) return MOE_ERR_INVALID_ARG;
  if (dims->d > 8192) return MOE_ERR_UNSUPPORTED;
  if (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) return MOE_ERR_INVALID_ARG;
  if ((st = check_weights(dims, weights)) != MOE_OK) return st;
  if ((st = check_ws(dims, ws, ws_bytes)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = cuda_status(launch_pre_norm(resid, pre_gain, eps, x, dims->T, dims->d, s))) != MOE_OK) return st;
  const ResidualArgs res{post_gain, eps, step, resid};
  return forward_impl(dims, x, w_r, sel_bias, weights, nullptr, &res, topk_idx, counts, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- dense SwiGLU MLP

// One expert, every token: the expert GEMMs with offsets {0, T}.
moe_dims_t dense_dims(const moe_dims_t& d) {
  moe_dims_t e = d;
  e.E = 1;
  e.n_groups = 1;
  e.topk_groups = 1;
  e.top_k = 1;
  e.routed_scale = 1.0f;
  return e;
}

moe_status_t check_dense_dims(const moe_dims_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->d <= 0 || d->inter <= 0) return MOE_ERR_INVALID_ARG;
  if (d->wfmt != MOE_W_BF16 && d->wfmt != MOE_W_NVFP4 && d->wfmt != MOE_W_FP8) return MOE_ERR_INVALID_ARG;
  if (d->T > 4194304 || d->d % 64 || d->inter % 64 || d->d > 16384 || d->inter > 65536) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

struct DenseLayout {
  size_t offs, table, tilex, h, total;
};

DenseLayout make_dense_layout(const moe_dims_t& d) {
  const ExpertPlan pl = plan_experts(d.T, d.d, 1, 1, d.inter, d.wfmt != MOE_W_BF16);
  DenseLayout L;
  size_t o = align_up(sizeof(WsHeader));
  L.offs = o;
  o = align_up(o + 2 * sizeof(int32_t));
  L.table = o;
  o = align_up(o + sizeof(int4));
  L.tilex = o;
  o = align_up(o + sizeof(int32_t) * static_cast<size_t>(pl.max_tiles));
  L.h = o;
  o = align_up(o + sizeof(uint16_t) * static_cast<size_t>(d.T) * d.inter);
  L.total = o;
  return L;
}

__global__ void dense_offsets_kernel(int32_t* offsets, int T) {
  pdl_launch_dependents();
  pdl_wait();
  offsets[0] = 0;
  offsets[1] = T;
}

moe_status_t moe_get_device_status(void* ws, void* stream, int32_t clear, int32_t* code) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  if (clear) {
    if (cudaMemsetAsync(ws, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t moe_set_stage_events(void* const* events, int32_t n) {
  if (!events || n < 6) {
    g_stage_events_on = false;
    return MOE_OK;
  }
  for (int i = 0; i < 6; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 6; ++i) g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_stage_events_on = true;
  return MOE_OK;
}

void moe_set_wait_bound(int64_t spins) { g_wait_spins = spins > 0 ? spins : kDefaultSpins; }

size_t moe_dense_workspace_bytes(const moe_dims_t* dims) {
  if (check_dense_dims(dims) != MOE_OK) return 0;
  return make_dense_layout(*dims).total;
}

moe_status_t moe_dense_mlp(const moe_dims_t* dims, const moe_bf16_t* x, const moe_expert_weights_t* w,
                           moe_bf16_t* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_dense_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const moe_dims_t d1 = dense_dims(*dims);
  if ((st = check_weights(&d1, w)) != MOE_OK) return st;
  const DenseLayout L = make_dense_layout(*dims);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* offs = reinterpret_cast<int32_t*>(base + L.offs);
  if (mark(0, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_pdl(dense_offsets_kernel, dim3(1), dim3(1), 0, s, offs, dims->T) != cudaSuccess) return MOE_ERR_CUDA;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  ExpertBuffers b{};
  b.x_perm = x;  // one expert: the permuted rows are the tokens in order
  b.offsets = offs;
  b.h = reinterpret_cast<uint16_t*>(base + L.h);
  b.y = out;
  b.y_f32 = nullptr;
  b.table = reinterpret_cast<int4*>(base + L.table);
  b.tile_expert = reinterpret_cast<int32_t*>(base + L.tilex);
  b.n_items = hdr->n_items;
  b.status = &hdr->status;
  b.timeout_where = &hdr->timeout_where;
  const ExpertWeightsDev wd = weights_dev(d1.wfmt, w);
  const ExpertPlan pl = plan_experts(d1.T, d1.d, 1, 1, d1.inter, d1.wfmt != MOE_W_BF16);
  int cu_error = 0;
  const cudaError_t e = launch_expert_ffn(pl, b, wd, d1.T, d1.d, 1, 1, d1.inter, num_sms(), g_wait_spins, s,
                                          &cu_error, g_stage_events_on ? g_stage_events[3] : nullptr);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return mark(4, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

const char* moe_version(void) { return "beammoe 0.1 sm_103a (tcgen05 bf16 grouped SwiGLU)"; }

}  // extern "C"
