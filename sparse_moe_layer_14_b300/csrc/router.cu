// Router of the Beam MoE block (release article, section "Mixture of
// Experts": sigmoid scores over all experts, groups ranked by the sum of
// their two best scores, the best groups kept, the top experts inside them
// chosen, weights normalised then scaled by 2.5; FP32 router per section
// "Residual stream").
//
// Small batches (decode):
//  router_simt_kernel    FP32 FMA logits = x . W_r for 64 tokens x 16 experts
//                        x one eighth of the hidden dimension per CTA, the
//                        eight CTAs of a split forming a cluster that adds its
//                        partials in a fixed order through distributed shared
//                        memory; the last CTA of each 8-token group (a ticket
//                        in the workspace header) then selects those tokens,
//                        one warp each: sigmoid, group top-2 sums, top groups,
//                        top experts, normalisation.
//  router_select_kernel  the same selection as its own kernel, for batches
//                        with more token groups than tickets.
//  wr_pad_kernel         a W_r copy with rows padded to a multiple of 4
//                        experts (tensor copies need 16-byte row strides).
// Large batches (prefill):
//  wr_split_kernel       W_r (fp32, [d][E]) -> three bf16 matrices hi, mid,
//                        lo ([E_pad][d], K-contiguous) with hi + mid + lo = W_r
//                        (8 + 8 + 8 significant bits cover fp32's 24), and the
//                        largest column norm of W_r (a fixed-order reduction).
//  router_tc_kernel      per 128 tokens and one range of the hidden dimension:
//                        partial logits x.hi + x.mid + x.lo on the tcgen05
//                        tensor cores (x is exact in bf16, so every product is
//                        exact in fp32); clusters of four token tiles share
//                        each W_r tile by TMA multicast.
//  router_select_flag_kernel  one warp per token: partials summed, sigmoid,
//                        group-limited selection and the two decision margins.
//                        The tensor cores' fp32 accumulation is coarser than
//                        FFMA, so a decision is kept only where every margin
//                        exceeds a bound on the logit error that scales with
//                        the token: kappa * 2^-23 * sqrt(d/16) * |x_t| *
//                        max_e |W_r[:, e]| (every partial sum of x_t . W_r[:, e]
//                        is at most |x_t| |W_r[:, e]| by Cauchy-Schwarz, and
//                        d/16 MMA steps each round once; kappa is set from
//                        measured errors with a wide margin). |x_t| is summed
//                        by the selecting warp from the token's row, the
//                        column norms of W_r come from wr_split_kernel.
//                        Elsewhere:
//  router_flagged_logits_kernel, router_flagged_select_kernel: tokens with a
//                        narrow margin get all logits in fp32 FFMA and the
//                        full warp selection.
#include <algorithm>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace cg = cooperative_groups;

namespace {

// Selection keys: an order-preserving map of a float score to an unsigned
// integer (a larger score gives a larger key; -0 and +0 share a key), so the
// warp finds a maximum with one redux.sync instead of a shuffle tree. Key 0
// is below every number's key and marks "no candidate" (experts outside the
// kept groups, taken ones, padding); a NaN score also maps to 0 and is never
// chosen.
__device__ __forceinline__ uint32_t score_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (v != v) return 0u;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kMaxPerLane = 8;  // E <= 256
constexpr uint32_t kFull = 0xffffffffu;

// Group-limited selection of one token by one warp. Lane l holds the scores
// of experts l, l+32, l+64, ... in s_in[] (entries of experts >= E are
// ignored); `bias` ([E] fp32, nullable) is the per-expert selection bias of
// DeepSeek-V3-style balancing: groups and experts are chosen on s + bias, the
// weights use s. Every choice takes the larger selection score, ties to the
// lower index. Writes the token's K expert ids (slot order: descending
// selection score) and weights scale * s_e / sum of the chosen s (summed in
// slot order). Returns, in every lane, the decision margins (on selection
// scores): x = worst kept group score - best dropped one; y = the smaller of
// (worst chosen score - best unchosen candidate) and the gaps between
// consecutive slots (1 where there is nothing to compare).
__device__ float2 warp_select(const float (&s_in)[kMaxPerLane], const float* __restrict__ bias, int lane, int t,
                              int E, int G, int Gk, int K, float scale, int32_t* __restrict__ topk_idx,
                              float* __restrict__ topk_w, int32_t* status) {
  const int gsz = E / G;
  uint32_t sk[kMaxPerLane];  // selection keys
  int grp[kMaxPerLane];      // group of each of this lane's experts (32 = none)
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    sk[i] = (e < E) ? score_key(bias ? s_in[i] + bias[e] : s_in[i]) : 0u;
    grp[i] = (e < E) ? e / gsz : 32;
  }

  uint32_t kept = 0u;
  float margin_group = 1.0f;
  if (gsz == 32) {
    // Groups of 32 (the Beam shape): element i of every lane is group i, so
    // all group scores come from independent warp reductions and end up in
    // every lane; the kept groups are then ranked without further exchange.
    uint32_t gk[kMaxPerLane];  // group score keys (0 past the last group)
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const uint32_t m1 = __reduce_max_sync(kFull, sk[i]);
      const int first = __ffs(__ballot_sync(kFull, sk[i] == m1)) - 1;  // a lane holding the largest
      const uint32_t m2 = __reduce_max_sync(kFull, lane == first ? 0u : sk[i]);
      gk[i] = i < G ? score_key(key_score(m1) + key_score(m2)) : 0u;
    }
    uint32_t last_kept = 0xffffffffu, best_dropped = 0u;
#pragma unroll
    for (int g = 0; g < kMaxPerLane; ++g) {
      if (g >= G) continue;
      int rank = 0;  // groups ahead of g: larger score, ties to the lower index
#pragma unroll
      for (int h = 0; h < kMaxPerLane; ++h)
        if (h < G && (gk[h] > gk[g] || (gk[h] == gk[g] && h < g))) ++rank;
      if (rank < Gk) {
        kept |= 1u << g;
        last_kept = min(last_kept, gk[g]);
      } else {
        best_dropped = max(best_dropped, gk[g]);
      }
    }
    if (Gk < G && best_dropped != 0u && last_kept != 0u) margin_group = key_score(last_kept) - key_score(best_dropped);
  } else {
    // group score = sum of the group's two largest selection scores (the
    // largest alone for one-expert groups); lane g keeps group g's
    float my_gs = 0.f;
#pragma unroll 4
    for (int g = 0; g < G; ++g) {
      uint32_t k1 = 0u, k2 = 0u;  // this lane's two largest keys in group g
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        if (grp[i] == g) {
          const uint32_t k = sk[i];
          k2 = max(k2, min(k1, k));
          k1 = max(k1, k);
        }
      }
      const uint32_t m1 = __reduce_max_sync(kFull, k1);
      const int first = __ffs(__ballot_sync(kFull, k1 == m1)) - 1;  // a lane holding the largest
      const uint32_t m2 = __reduce_max_sync(kFull, lane == first ? k2 : k1);
      if (lane == g) my_gs = gsz >= 2 ? key_score(m1) + key_score(m2) : key_score(m1);
    }

    // keep the Gk best groups
    const bool is_group = lane < G;
    const uint32_t gkey = is_group ? score_key(my_gs) : 0u;
    uint32_t last_kept = 0u;
    for (int r = 0; r < Gk; ++r) {
      const bool cand = is_group && !((kept >> lane) & 1u);
      const uint32_t m = __reduce_max_sync(kFull, cand ? gkey : 0u);
      const uint32_t w = __reduce_min_sync(kFull, (cand && gkey == m) ? static_cast<uint32_t>(lane) : 32u);
      if (w < 32u) kept |= 1u << w;
      last_kept = m;
    }
    if (Gk < G) {
      const bool cand = is_group && !((kept >> lane) & 1u);
      const uint32_t m = __reduce_max_sync(kFull, cand ? gkey : 0u);
      if (m != 0u && last_kept != 0u) margin_group = key_score(last_kept) - key_score(m);
    }
  }

  // choose the K best experts of the kept groups
  uint32_t ck[kMaxPerLane];  // candidate keys (0 once taken or outside the kept groups)
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) ck[i] = (grp[i] < 32 && ((kept >> grp[i]) & 1u)) ? sk[i] : 0u;
  float my_w = 0.f;  // slot `lane`: its unbiased score
  int my_e = 0;      // ... and its expert
  float sum = 0.f;   // of unbiased scores, in slot order
  float prev = 0.f, gap = 1.0f;
  for (int k = 0; k < K; ++k) {
    uint32_t kb = 0u;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) kb = max(kb, ck[i]);
    uint32_t eb = 0xffffffffu;  // lowest expert of this lane holding kb
#pragma unroll
    for (int i = kMaxPerLane - 1; i >= 0; --i)
      if (ck[i] == kb) eb = static_cast<uint32_t>(lane + 32 * i);
    const uint32_t m = __reduce_max_sync(kFull, kb);
    const uint32_t idx = __reduce_min_sync(kFull, (kb == m && m != 0u) ? eb : 0xffffffffu);
    float u = 0.f, v = 0.f;
    int e = 0;
    if (m == 0u || idx >= static_cast<uint32_t>(E)) {  // fewer than K candidates (NaN scores)
      latch_status(status, MOE_DEV_BAD_EXPERT);
    } else {
      e = static_cast<int>(idx);
      v = key_score(m);
      const int owner = e & 31, slot = e >> 5;
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        if (i == slot) {
          mine = s_in[i];
          if (lane == owner) ck[i] = 0u;
        }
      }
      u = __shfl_sync(kFull, mine, owner);
    }
    sum += u;
    if (k > 0) gap = fminf(gap, prev - v);
    prev = v;
    if (lane == k) {
      my_w = u;
      my_e = e;
    }
  }
  float margin = gap;
  {
    uint32_t kb = 0u;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) kb = max(kb, ck[i]);
    const uint32_t m = __reduce_max_sync(kFull, kb);
    if (m != 0u) margin = fminf(margin, prev - key_score(m));
  }
  if (lane < K) {
    float w = 0.f;
    if (sum > 0.f) {
      w = scale * my_w / sum;
    } else if (lane == 0) {
      latch_status(status, MOE_DEV_ZERO_SUM);
    }
    topk_idx[static_cast<size_t>(t) * K + lane] = my_e;
    topk_w[static_cast<size_t>(t) * K + lane] = w;
  }
  return make_float2(margin_group, margin);
}

__device__ __forceinline__ float sigmoid(float l) { return 1.0f / (1.0f + expf(-l)); }

// One warp per token: sigmoid of the final logits [T][E] and the selection
// (used where the fused router below cannot select itself).
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits, int T,
                                                            int E, int G, int Gk, int K, float scale,
                                                            const float* __restrict__ bias,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ topk_w, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  float s[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = (e < E) ? sigmoid(logits[static_cast<size_t>(t) * E + e]) : 0.f;
  }
  warp_select(s, bias, lane, t, E, G, Gk, K, scale, topk_idx, topk_w, status);
}

// ---------------------------------------------------------------- SIMT path (small batches)
//
// router_simt_kernel: one CTA per (64 tokens, 16 experts, 1/8 of the hidden
// dimension); the 8 CTAs of a hidden-dimension split form a thread-block
// cluster. A producer warp streams x (bf16, 128-byte swizzled rows) and W_r
// (fp32) tiles of 64 hidden elements through an 8-deep shared-memory ring by
// TMA; each of 8 consumer warps takes 8 of a stage's 64 hidden elements for
// the whole 64 x 16 tile (lane: 4 tokens x 8 experts, packed FP32 FMAs). The
// partial sums are added in a fixed order: the warps' in the CTA, then the
// cluster's CTAs through distributed shared memory, each CTA finishing 8 of
// the 64 tokens, so the logits do not depend on scheduling. They go to
// logits[T][E]. The last CTA to finish a group of 8 tokens (counted in a
// ticket that it returns to 0) then selects those tokens, one warp each.

constexpr int kRsTokens = 64;    // tokens per tile
constexpr int kRsExperts = 16;   // experts per tile
constexpr int kRsBK = 64;        // hidden elements per pipeline stage
constexpr int kRsCluster = 8;    // CTAs per cluster: parts of the hidden dimension
constexpr int kRsStages = 8;
constexpr int kRsWarps = 8;      // consumer warps; one more warp produces
constexpr int kRsThreads = 32 * (kRsWarps + 1);
constexpr int kRsTokensPerRank = kRsTokens / kRsCluster;  // tokens each CTA finishes (and may select)
constexpr uint32_t kRsXBytes = kRsTokens * kRsBK * 2;     // 8 KB
constexpr uint32_t kRsWBytes = kRsBK * kRsExperts * 4;    // 4 KB
constexpr uint32_t kRsStageBytes = kRsXBytes + kRsWBytes; // 12 KB, a multiple of 1024
constexpr uint64_t kRsWaitNs = 2000000000ull;
constexpr uint64_t kRsDrainNs = 1000000000ull;
static_assert(kRsWarps * 8 == kRsBK, "a consumer warp takes 8 hidden elements of a stage");
static_assert(kRsTokens * kRsExperts == 4 * 256 && kRsTokensPerRank * kRsExperts == 128, "reduction shapes");

struct RsArgs {
  int T, d, E, G, Gk, K;
  float scale;
  const float* bias;   // [E] selection bias or null
  float* logits;       // [T][E]
  int32_t* ticket;     // [ceil(T / 64) * 8], zero between calls; null: the selection runs separately
  int32_t* topk_idx;
  float* topk_w;
  int32_t* status;
  int32_t* timeout_where;
  long long wait_spins;
};

// d = (a, a) * b + c, two IEEE fp32 FMAs in one instruction
__device__ __forceinline__ float2 fma2(float a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %2};\n mov.b64 rb, {%3, %4};\n mov.b64 rc, {%5, %6};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ void rs_fail(const RsArgs& a, volatile int* abort, int where) {
  latch_status(a.status, MOE_DEV_TIMEOUT);
  if (a.timeout_where) atomicCAS(a.timeout_where, 0, where);
  *abort = 1;
}

__global__ void __cluster_dims__(1, 1, kRsCluster) __launch_bounds__(kRsThreads, 2)
    router_simt_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const RsArgs a) {
  extern __shared__ uint8_t rs_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRsStages];
  __shared__ __align__(8) uint64_t empty_bar[kRsStages];
  __shared__ __align__(16) float cta_part[kRsTokens * kRsExperts];  // this CTA's sums, [token][expert]
  __shared__ int abort_flag, is_last;
  uint8_t* smem = rs_raw + ((1024u - (smem_u32(rs_raw) & 1023u)) & 1023u);
  volatile int* abort = &abort_flag;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRsTokens, e0 = blockIdx.y * kRsExperts;
  const int nchunks = a.d / kRsBK;
  const int c0 = rank * nchunks / kRsCluster, c1 = (rank + 1) * nchunks / kRsCluster;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRsStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kRsWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kRsWarps && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  __syncthreads();
  pdl_wait();  // x may come from earlier work on the stream

  int issued = 0;
  const int q = lane & 15, o = lane >> 4;  // tokens q, q+16, q+32, q+48; experts 8o .. 8o+7
  float2 acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 4; ++p) acc[j][p] = make_float2(0.f, 0.f);
  if (warp == kRsWarps) {
    if (lane == 0) {
      for (int i = 0; i < c1 - c0; ++i) {
        const int s = i % kRsStages;
        if (i >= kRsStages &&
            !mbar_wait_bounded(&empty_bar[s], static_cast<uint32_t>((i / kRsStages - 1) & 1), a.wait_spins, kRsWaitNs,
                               abort)) {
          if (!*abort) rs_fail(a, abort, 15);
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * kRsStageBytes;
        mbar_arrive_expect_tx(&full_bar[s], kRsStageBytes);
        tma_load_2d(st, &tmX, (c0 + i) * kRsBK, t0, &full_bar[s]);
        tma_load_2d(st + kRsXBytes, &tmW, e0, (c0 + i) * kRsBK, &full_bar[s]);
        ++issued;
      }
    }
  } else {
    for (int i = 0; i < c1 - c0; ++i) {
      const int s = i % kRsStages;
      const bool ok =
          __all_sync(kFull, mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((i / kRsStages) & 1), a.wait_spins,
                                              kRsWaitNs, abort));
      if (!ok) {
        if (lane == 0 && !*abort) rs_fail(a, abort, 16);
        break;
      }
      const uint8_t* st = smem + static_cast<size_t>(s) * kRsStageBytes;
      const float* ws = reinterpret_cast<const float*>(st + kRsXBytes) + warp * 8 * kRsExperts + o * 8;
      uint4 xv[4];  // x[t][8 warp .. 8 warp + 7] of the lane's tokens (16-byte chunk `warp` of a swizzled row)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = q + 16 * j;
        xv[j] = *reinterpret_cast<const uint4*>(st + t * 128 + ((warp ^ (t & 7)) << 4));
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const float4 w0 = *reinterpret_cast<const float4*>(ws + kk * kRsExperts);
        const float4 w1 = *reinterpret_cast<const float4*>(ws + kk * kRsExperts + 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t word = (&xv[j].x)[kk >> 1];
          const float xf = __uint_as_float((kk & 1) ? (word & 0xFFFF0000u) : (word << 16));
          acc[j][0] = fma2(xf, make_float2(w0.x, w0.y), acc[j][0]);
          acc[j][1] = fma2(xf, make_float2(w0.z, w0.w), acc[j][1]);
          acc[j][2] = fma2(xf, make_float2(w1.x, w1.y), acc[j][2]);
          acc[j][3] = fma2(xf, make_float2(w1.z, w1.w), acc[j][3]);
        }
      }
      fence_proxy_async_smem();  // the reads above complete before TMA may refill the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }
  __syncthreads();

  // the warps' partial tiles, added in warp order (the ring is free: every
  // stage was consumed unless the CTA gave up, and then nothing is reused)
  const bool aborted = *abort != 0;
  float* red = reinterpret_cast<float*>(smem);  // [warp][token][expert]
  if (!aborted && warp < kRsWarps) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float* row = red + (warp * kRsTokens + q + 16 * j) * kRsExperts + o * 8;
      *reinterpret_cast<float4*>(row) = make_float4(acc[j][0].x, acc[j][0].y, acc[j][1].x, acc[j][1].y);
      *reinterpret_cast<float4*>(row + 4) = make_float4(acc[j][2].x, acc[j][2].y, acc[j][3].x, acc[j][3].y);
    }
  }
  __syncthreads();
  if (!aborted && threadIdx.x < 256) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i = threadIdx.x + 256 * m;
      float v = red[i];
#pragma unroll
      for (int w = 1; w < kRsWarps; ++w) v += red[w * kRsTokens * kRsExperts + i];
      cta_part[i] = v;
    }
  }
  cluster.sync();  // every CTA's partial tile is published

  // this CTA finishes tokens t0 + 8 rank .. + 7: the cluster's partials in rank order
  if (threadIdx.x < kRsTokensPerRank * kRsExperts) {
    const int i = rank * kRsTokensPerRank * kRsExperts + threadIdx.x;
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < kRsCluster; ++c) v += cluster.map_shared_rank(cta_part, c)[i];
    const int t = t0 + i / kRsExperts, e = e0 + i % kRsExperts;
    if (t < a.T && e < a.E) a.logits[static_cast<size_t>(t) * a.E + e] = v;
    __threadfence();
  }
  cluster.sync();  // no CTA leaves while another may still read its partials

  if (aborted && warp == kRsWarps && lane == 0) {
    // some waits returned early: let every copy issued into each stage land
    // (bounded) before the CTA exits
    for (int s = 0; s < kRsStages; ++s) {
      if (issued > s) {
        const int f = s + kRsStages * ((issued - 1 - s) / kRsStages);
        mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((f / kRsStages) & 1), 1ll << 40, kRsDrainNs, nullptr);
      }
    }
  }
  if (a.ticket == nullptr) return;
  if (threadIdx.x == 0) {
    int32_t* tk = a.ticket + blockIdx.x * kRsCluster + rank;
    is_last = atomicAdd(tk, 1) == static_cast<int>(gridDim.y) - 1;
    if (is_last) *tk = 0;  // every CTA of this call has counted: ready for the next call
  }
  __syncthreads();
  if (!is_last || warp >= kRsTokensPerRank) return;
  __threadfence();
  const int t = t0 + rank * kRsTokensPerRank + warp;
  if (t >= a.T) return;
  float s[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = (e < a.E) ? sigmoid(__ldcg(a.logits + static_cast<size_t>(t) * a.E + e)) : 0.f;
  }
  warp_select(s, a.bias, lane, t, a.E, a.G, a.Gk, a.K, a.scale, a.topk_idx, a.topk_w, a.status);
}

// W_r [d][E] -> [d][E4] (E4 = E rounded up to a multiple of 4, zero columns
// added), so its rows meet the 16-byte stride rule of tensor copies.
__global__ void __launch_bounds__(256) wr_pad_kernel(const float* __restrict__ wr, int d, int E, int E4,
                                                     float* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t n = static_cast<int64_t>(d) * E4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = i / E4;
    const int e = static_cast<int>(i - k * E4);
    out[i] = e < E ? wr[k * E + e] : 0.f;
  }
}

// ---------------------------------------------------------------- tensor-core path

// tma_load_2d into the same shared-memory offset of every CTA of the cluster
// named in `mask` (bit i: the CTA of cluster rank i), completion counted on
// the mbarrier at `bar`'s offset in each of them.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                                      uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, "
      "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// mma_commit arriving on the mbarrier at `bar`'s offset in every CTA of the
// cluster named in `mask`.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}


// Shared-memory matrix descriptor of a K-major bf16 tile with 64-byte rows
// and the 64-byte swizzle (8-row atoms of 512 bytes): start address >> 4,
// leading offset 1 (unused when swizzled), stride 512 >> 4 between 8-row
// groups, descriptor version 1 (bit 46), layout type 4 (64-byte swizzle).
// A 16-wide K step (32 bytes) adds 2 to the start address field.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(512u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(4u) << 61;
  return d;
}

constexpr int kTcTokens = 128;  // tokens per CTA (MMA M)
constexpr int kTcBK = 32;       // hidden elements per pipeline stage (64-byte rows, 64-byte swizzle)
constexpr int kTcStages = 4;
constexpr int kTcMaxSplits = 16;
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint64_t kTcDrainNs = 1000000000ull;

// out[s][e][k] = bf16 split s of W_r[k][e] (rows e >= E are zero). Also
// resets the flagged-token count, and finds the largest column norm of W_r in
// a fixed order: every block (128 hidden rows x 32 experts) writes the sums of
// squares of its columns to colss[k block][e]; the last block to finish a
// 32-expert strip (counted in ticket[strip], which it returns to 0) adds them
// up in k order and writes the strip's largest norm to wn_strip[strip]. A
// thread splits 16 consecutive hidden elements of one expert, so each plane
// is written in 32-byte pieces (eight threads: 256 contiguous bytes).
constexpr int kWsRows = 128;  // hidden rows per wr_split block (d is a multiple of 256 on this path)

__device__ __forceinline__ uint32_t bf16_pair(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

__global__ void __launch_bounds__(256) wr_split_kernel(const float* __restrict__ wr, int d, int E, int E_pad,
                                                       uint16_t* __restrict__ out, float* __restrict__ colss,
                                                       float* __restrict__ wn_strip, int32_t* __restrict__ ticket,
                                                       int32_t* __restrict__ flagged_count) {
  __shared__ float tile[kWsRows][33];
  __shared__ int is_last;
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *flagged_count = 0;
  const int k0 = blockIdx.x * kWsRows, e0 = blockIdx.y * 32;
  const int E32 = gridDim.y * 32;  // row stride of colss
  {
    const int c = (threadIdx.x & 7) * 4;  // 8 threads read one 128-byte row piece
#pragma unroll
    for (int j = 0; j < kWsRows / 32; ++j) {
      const int r = (threadIdx.x >> 3) + 32 * j;
      const float* src = wr + static_cast<size_t>(k0 + r) * E + e0 + c;
#pragma unroll
      for (int q = 0; q < 4; ++q) tile[r][c + q] = (e0 + c + q < E) ? src[q] : 0.f;
    }
  }
  __syncthreads();
  const int e = threadIdx.x >> 3, kc = threadIdx.x & 7;  // expert e0 + e, hidden rows 16 kc .. 16 kc + 15
  uint32_t hi[8], mid[8], lo[8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    __nv_bfloat16 h[2], m[2], l[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float w = tile[kc * 16 + i + u][e];
      ss = fmaf(w, w, ss);
      h[u] = __float2bfloat16_rn(w);
      const float r1 = w - __bfloat162float(h[u]);
      m[u] = __float2bfloat16_rn(r1);
      l[u] = __float2bfloat16_rn(r1 - __bfloat162float(m[u]));
    }
    hi[i / 2] = bf16_pair(h[0], h[1]);
    mid[i / 2] = bf16_pair(m[0], m[1]);
    lo[i / 2] = bf16_pair(l[0], l[1]);
  }
  // the 8 threads of an expert are 8 consecutive lanes: pairwise sums in a fixed order
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, off, 8);
  if (kc == 0) colss[static_cast<size_t>(blockIdx.x) * E32 + e0 + e] = ss;
  if (e0 + e < E_pad) {
    const size_t o = static_cast<size_t>(e0 + e) * d + k0 + kc * 16;
    const size_t plane = static_cast<size_t>(E_pad) * d;
    uint4* dh = reinterpret_cast<uint4*>(out + o);
    uint4* dm = reinterpret_cast<uint4*>(out + plane + o);
    uint4* dl = reinterpret_cast<uint4*>(out + 2 * plane + o);
    dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    dm[0] = make_uint4(mid[0], mid[1], mid[2], mid[3]);
    dm[1] = make_uint4(mid[4], mid[5], mid[6], mid[7]);
    dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
  __threadfence();  // this block's column sums are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&ticket[blockIdx.y], 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (is_last && threadIdx.x < 32) {
    const int tx = threadIdx.x;
    float cs = 0.f;
    for (int kx = 0; kx < static_cast<int>(gridDim.x); ++kx) cs += __ldcg(colss + static_cast<size_t>(kx) * E32 + e0 + tx);
    float nrm = sqrtf(cs);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) nrm = fmaxf(nrm, __shfl_xor_sync(0xffffffffu, nrm, off));
    if (tx == 0) {
      wn_strip[blockIdx.y] = nrm;
      ticket[blockIdx.y] = 0;
    }
  }
}

struct TcArgs {
  int T, d, E, E_pad;
  int kb_per_split;  // K slices of one CTA (the hidden dimension is split over blockIdx.y)
  float* part;       // [splits][T][E] partial logits
  int32_t* status;
  int32_t* timeout_where;
  long long wait_spins;
  uint32_t stage_bytes;
  uint32_t tmem_cols;
  int cluster;       // CTAs of a cluster (consecutive token tiles, one hidden range): 1, 2 or 4
};

__device__ __forceinline__ void tc_fail(const TcArgs& a, volatile int* abort, int where) {
  latch_status(a.status, MOE_DEV_TIMEOUT);
  if (a.timeout_where) atomicCAS(a.timeout_where, 0, where);
  *abort = 1;
}

// Partial logits of 128 tokens x E_pad experts over one range of the hidden
// dimension: hi products accumulate in D1 (TMEM columns [0, E_pad)), the small
// mid and lo products in D2 ([E_pad, 2 E_pad)), so they keep their bits.
// The CTAs of a cluster share their hidden range: each loads 1/cluster of
// every split-W_r tile and multicasts it to all of them (W_r is read from L2
// once per cluster, not once per CTA), so a stage is refilled only after every
// CTA of the cluster has consumed it (each MMA issuer's commit arrives on the
// stage's empty barrier in every CTA).
__global__ void __launch_bounds__(192, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const __grid_constant__ CUtensorMap tmW, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTcStages];
  __shared__ __align__(8) uint64_t empty_bar[kTcStages];
  __shared__ __align__(8) uint64_t accf_bar;
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
  pdl_launch_dependents();
  const int t0 = blockIdx.x * kTcTokens;
  const int kb0 = blockIdx.y * a.kb_per_split, kb1 = kb0 + a.kb_per_split;
  const uint32_t wtile = static_cast<uint32_t>(a.E_pad) * kTcBK * 2;  // one split's tile
  constexpr uint32_t kXTile = kTcTokens * kTcBK * 2;                  // 8 KB
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const uint16_t cmask = static_cast<uint16_t>((1u << a.cluster) - 1u);
  const int part_rows = a.E_pad / a.cluster;                         // W_r rows this CTA loads
  const uint32_t part_off = static_cast<uint32_t>(crank * part_rows) * kTcBK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], a.cluster);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster.sync();  // every CTA's barriers are initialised before any multicast or remote arrival
  tc_fence_after();
  pdl_wait();  // x and the split W_r come from earlier work on the stream
  const uint32_t tmem_base = tmem_slot;
  long long fills = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, a.wait_spins, kTcWaitNs, abort)) {
          if (!*abort) tc_fail(a, abort, 11);
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(stage) * a.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[stage], kXTile + 3 * wtile);
        tma_load_2d(st, &tmX, kb * kTcBK, t0, &full_bar[stage]);
        for (int sp = 0; sp < 3; ++sp) {
          uint8_t* dst = st + kXTile + sp * wtile + part_off;
          const int row = sp * a.E_pad + crank * part_rows;
          if (a.cluster > 1) {
            tma_load_2d_multicast(dst, &tmW, kb * kTcBK, row, &full_bar[stage], cmask);
          } else {
            tma_load_2d(dst, &tmW, kb * kTcBK, row, &full_bar[stage]);
          }
        }
        ++fills;
        if (++stage == kTcStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t idesc = idesc_bf16_f32(kTcTokens, a.E_pad);
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, a.wait_spins, kTcWaitNs, abort)) {
          if (!*abort) tc_fail(a, abort, 12);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sx = smem_u32(smem + static_cast<size_t>(stage) * a.stage_bytes);
#pragma unroll
        for (int k = 0; k < kTcBK / 16; ++k) {
          const uint64_t adesc = sdesc_kmajor_sw64(sx + k * 32);
          const uint32_t first = ((kb - kb0) | k) != 0 ? 1u : 0u;
          mma_bf16_ss(tmem_base, adesc, sdesc_kmajor_sw64(sx + kXTile + k * 32), idesc, first);
          mma_bf16_ss(tmem_base + a.E_pad, adesc, sdesc_kmajor_sw64(sx + kXTile + wtile + k * 32), idesc, first);
          mma_bf16_ss(tmem_base + a.E_pad, adesc, sdesc_kmajor_sw64(sx + kXTile + 2 * wtile + k * 32), idesc, 1u);
        }
        // the last kTcStages stages are not refilled: no release (and no late remote arrival)
        if (kb + kTcStages < kb1) {
          if (a.cluster > 1) {
            mma_commit_multicast(&empty_bar[stage], cmask);
          } else {
            mma_commit(&empty_bar[stage]);
          }
        }
        if (++stage == kTcStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(&accf_bar);
    }
    __syncwarp();
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (tokens t0 + 32 q ..): the partial logits go to global
    const int q = warp & 3;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&accf_bar, 0, a.wait_spins, kTcWaitNs, abort));
    if (ok) {
      // 32 columns at a time: D1 + D2 of this thread's token into a padded
      // 32 x 32 shared tile (the ring is free once the MMAs are done), then
      // written out token by token with the lanes along the columns, so each
      // store covers 128 contiguous bytes of one row.
      tc_fence_after();
      float* sm = reinterpret_cast<float*>(smem) + q * 32 * 33;
      float* dst0 = a.part + (static_cast<size_t>(blockIdx.y) * a.T + t0 + q * 32) * a.E;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      for (int c = 0; c < a.E_pad; c += 32) {
        const bool two = c + 16 < a.E_pad;  // both 16-column halves lie inside the accumulators
        uint32_t v[16], v2[16], w[16], w2[16];
        tmem_ld_32x32b_x16(tb + c, v);
        tmem_ld_32x32b_x16(tb + a.E_pad + c, v2);
        if (two) {
          tmem_ld_32x32b_x16(tb + c + 16, w);
          tmem_ld_32x32b_x16(tb + a.E_pad + c + 16, w2);
        }
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          sm[lane * 33 + j] = __uint_as_float(v[j]) + __uint_as_float(v2[j]);
          sm[lane * 33 + 16 + j] = two ? __uint_as_float(w[j]) + __uint_as_float(w2[j]) : 0.f;
        }
        __syncwarp();
        for (int i = 0; i < 32; ++i) {
          if (t0 + q * 32 + i < a.T && c + lane < a.E) dst0[static_cast<size_t>(i) * a.E + c + lane] = sm[i * 33 + lane];
        }
        __syncwarp();
      }
    } else if (lane == 0 && !*abort) {
      tc_fail(a, abort, 13);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort) {
    if (threadIdx.x == 0) {
      for (int s = 0; s < kTcStages; ++s) {
        if (fills > s) {
          const long long f = s + static_cast<long long>(kTcStages) * ((fills - 1 - s) / kTcStages);
          mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((f / kTcStages) & 1), 1ll << 40, kTcDrainNs, nullptr);
        }
      }
    }
    if (warp == 1 && lane == 0) {
      mma_commit(&drain_bar);
      mbar_wait_bounded(&drain_bar, 0, 1ll << 40, kTcDrainNs, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (warp == 1) tmem_dealloc(tmem_base, a.tmem_cols);
  // No CTA leaves while a peer may still multicast into it or arrive on its
  // barriers. After a timeout a peer may have issued a copy for a stage that
  // this CTA no longer waits for: give such copies time to land (bounded).
  const bool aborted = *abort != 0;
  cluster.sync();
  if (aborted && a.cluster > 1 && threadIdx.x == 0) {
    const uint64_t t_end = globaltimer_ns() + 100000;
    while (globaltimer_ns() < t_end) __nanosleep(1000);
  }
}

// One warp per token: the tensor-core logits (partials summed in a fixed
// order), sigmoid, the group-limited selection and its weights. Where a
// decision margin (kept groups, chosen experts, slot order) could be within
// the tensor-core error of zero, the token is flagged for an fp32 recompute
// of all its logits; elsewhere the decisions equal those of exact fp32
// logits and only the weights carry the tensor-core error (about 1e-6
// relative).
//   logit error bound  e_l = err_coef * |x_t| * max_e |W_r[:, e]|,
//                      err_coef = kappa * 2^-23 * sqrt(d / 16)
//   score error bound  e_s = e_l / 4 (the sigmoid's slope is at most 1/4)
// A group score sums two scores and a group margin compares two group
// scores (4 e_s); expert margins and slot gaps compare two scores (2 e_s).
__global__ void __launch_bounds__(256) router_select_flag_kernel(const float* __restrict__ part, int splits, int T,
                                                                 int E, int G, int Gk, int K, float scale,
                                                                 const float* __restrict__ bias,
                                                                 const uint16_t* __restrict__ x, int d,
                                                                 const float* __restrict__ wn_strip, int n_strips,
                                                                 float err_coef, int32_t* __restrict__ topk_idx,
                                                                 float* __restrict__ topk_w,
                                                                 int32_t* __restrict__ flagged,
                                                                 int32_t* __restrict__ flagged_count,
                                                                 int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  float s[kMaxPerLane];
  float l[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) l[i] = 0.f;
  for (int sp = 0; sp < splits; ++sp) {  // eight independent loads per split, summed in split order
    const float* row = part + (static_cast<size_t>(sp) * T + t) * E;
    float v[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) v[i] = (lane + 32 * i < E) ? row[lane + 32 * i] : 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) l[i] += v[i];
  }
  // |x_t|^2 for the error bound: the warp reads the token's row (16-byte loads, lanes side by side)
  float xs = 0.f;
  {
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
    const int n16 = d / 8;  // 16-byte pieces of the row (d is a multiple of 256 on this path)
    for (int i0 = lane; i0 < n16; i0 += 4 * 32) {
      uint4 v[4];  // four loads in flight
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = i0 + 32 * u < n16 ? __ldg(xr + i0 + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(w4[j] << 16), hi = __uint_as_float(w4[j] & 0xFFFF0000u);
          xs = fmaf(lo, lo, xs);
          xs = fmaf(hi, hi, xs);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xs += __shfl_xor_sync(0xffffffffu, xs, off);
  }
  float wn = 0.f;
  for (int i = 0; i < n_strips; ++i) wn = fmaxf(wn, wn_strip[i]);
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = (e < E) ? sigmoid(l[i]) : 0.f;
  }
  const float2 margin = warp_select(s, bias, lane, t, E, G, Gk, K, scale, topk_idx, topk_w, status);
  const float e_s = 0.25f * err_coef * sqrtf(xs) * wn;
  const bool narrow = !(margin.x >= 4.f * e_s && margin.y >= 2.f * e_s);  // NaN margins are narrow too
  if (lane == 0 && narrow) flagged[atomicAdd(flagged_count, 1)] = t;
}

// Flagged tokens: every logit as an fp32 FFMA dot product. Work items are
// (group of up to kFlagTokens flagged tokens, one of `splits` parts of the
// hidden dimension: 16, or 8 where d is not a multiple of 16 x 32), taken
// round-robin by the CTAs; an item streams its rows of W_r
// through shared memory in chunks of kFlagRows rows by bulk-async copies (a
// 6-deep ring: the copy latency, not the FMAs, bounds an item), thread (q, e)
// of the 1024 adds rows q, q+4, ... of each chunk for expert e, and the four
// sums are added in a fixed order into the item's partial logits
// part[part][i][e].
constexpr int kFlagTokens = 4;
constexpr int kFlagThreads = 1024;
constexpr int kFlagRows = 32;    // W_r rows per chunk (32 x E fp32)
constexpr int kFlagRing = 6;
constexpr int kFlagSplits = kRouterFlagSplits;  // hidden-dimension parts per token group (at most)

int flag_splits(int d) { return d % (kFlagSplits * kFlagRows) == 0 ? kFlagSplits : kFlagSplits / 2; }

__global__ void __launch_bounds__(kFlagThreads) router_flagged_logits_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, int T, int d, int E,
    const int32_t* __restrict__ flagged, const int32_t* __restrict__ flagged_count, float* __restrict__ part_out,
    int splits, int32_t* status, int32_t* timeout_where, long long wait_spins) {
  extern __shared__ __align__(16) uint8_t fsm[];
  float4* xs4 = reinterpret_cast<float4*>(fsm);                      // [d / splits]: x of <= 4 tokens at k
  float* wring = reinterpret_cast<float*>(fsm + sizeof(float4) * (d / splits));  // [ring][rows][E]
  __shared__ float part[4][kFlagTokens][256];
  __shared__ __align__(8) uint64_t bar[kFlagRing];
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  pdl_launch_dependents();
  pdl_wait();
  const int n = *flagged_count;
  if (n == 0 || !dcheck(n <= T, status)) return;
  const int groups = (n + kFlagTokens - 1) / kFlagTokens;
  const int e = threadIdx.x & 255, q = threadIdx.x >> 8;
  const uint32_t chunk_bytes = static_cast<uint32_t>(kFlagRows) * E * sizeof(float);
  const int kq = d / splits;              // hidden elements of one item
  const int nchunks = kq / kFlagRows;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFlagRing; ++i) mbar_init(&bar[i], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t issued = 0, consumed = 0;  // chunk copies issued (thread 0) / waited
  for (int item = blockIdx.x; item < groups * splits; item += gridDim.x) {
    const int i0 = (item / splits) * kFlagTokens, z = item % splits;
    const int nt = min(kFlagTokens, n - i0);
    const int k0 = z * kq;
    const float* wsrc = wr + static_cast<size_t>(k0) * E;
    for (int k = threadIdx.x; k < kq; k += blockDim.x) {
      float v[kFlagTokens];
#pragma unroll
      for (int j = 0; j < kFlagTokens; ++j)
        v[j] = (j < nt && dcheck(flagged[i0 + j] >= 0 && flagged[i0 + j] < T, status))
                   ? bf16_bits_to_float(x[static_cast<size_t>(flagged[i0 + j]) * d + k0 + k])
                   : 0.f;
      xs4[k] = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (threadIdx.x == 0) {
      for (int c = 0; c < kFlagRing - 1 && c < nchunks; ++c) {
        const uint32_t slot = issued % kFlagRing;
        mbar_arrive_expect_tx(&bar[slot], chunk_bytes);
        bulk_load(wring + static_cast<size_t>(slot) * kFlagRows * E, wsrc + static_cast<size_t>(c) * kFlagRows * E,
                  chunk_bytes, &bar[slot]);
        ++issued;
      }
    }
    __syncthreads();
    float acc[kFlagTokens] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < nchunks; ++c) {
      if (threadIdx.x == 0 && c + kFlagRing - 1 < nchunks) {
        const uint32_t slot = issued % kFlagRing;  // its previous chunk was consumed before the last barrier
        mbar_arrive_expect_tx(&bar[slot], chunk_bytes);
        bulk_load(wring + static_cast<size_t>(slot) * kFlagRows * E,
                  wsrc + static_cast<size_t>(c + kFlagRing - 1) * kFlagRows * E, chunk_bytes, &bar[slot]);
        ++issued;
      }
      const uint32_t slot = consumed % kFlagRing;
      // On a timeout every later wait returns at once (the loop stays the same
      // for all threads, so the barriers below match); the status is latched.
      if (!mbar_wait_bounded(&bar[slot], (consumed / kFlagRing) & 1u, wait_spins, 2000000000ull, abort) && !*abort) {
        latch_status(status, MOE_DEV_TIMEOUT);
        if (timeout_where) atomicCAS(timeout_where, 0, 14);
        *abort = 1;
      }
      ++consumed;
      const float* wc = wring + static_cast<size_t>(slot) * kFlagRows * E;
      if (e < E) {
#pragma unroll
        for (int rr = q; rr < kFlagRows; rr += 4) {
          const float w = wc[rr * E + e];
          const float4 a = xs4[c * kFlagRows + rr];
          acc[0] = fmaf(a.x, w, acc[0]);
          acc[1] = fmaf(a.y, w, acc[1]);
          acc[2] = fmaf(a.z, w, acc[2]);
          acc[3] = fmaf(a.w, w, acc[3]);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();  // the slot may be refilled after every thread is done with it
    }
#pragma unroll
    for (int j = 0; j < kFlagTokens; ++j) part[q][j][e] = acc[j];
    __syncthreads();
    if (q == 0 && e < E) {
      for (int j = 0; j < nt; ++j)
        part_out[(static_cast<size_t>(z) * n + i0 + j) * E + e] =
            ((part[0][j][e] + part[1][j][e]) + part[2][j][e]) + part[3][j][e];
    }
    __syncthreads();
  }
  // After an abort some waits returned early: let every copy issued into each
  // slot land (bounded) before the CTA exits.
  if (*abort && threadIdx.x == 0) {
    for (uint32_t sl = 0; sl < kFlagRing; ++sl) {
      if (issued > sl) {
        const uint32_t f = sl + kFlagRing * ((issued - 1 - sl) / kFlagRing);
        mbar_wait_bounded(&bar[sl], (f / kFlagRing) & 1u, 1ll << 40, 1000000000ull, nullptr);
      }
    }
  }
  __syncthreads();
}

// One warp per flagged token: the parts' partial logits summed in order,
// sigmoid and the full selection.
__global__ void __launch_bounds__(256) router_flagged_select_kernel(const float* __restrict__ part, int splits, int T,
                                                                   int E,
                                                                   int G,
                                                                   int Gk, int K, float scale,
                                                                   const float* __restrict__ bias,
                                                                   const int32_t* __restrict__ flagged,
                                                                   const int32_t* __restrict__ flagged_count,
                                                                   int32_t* __restrict__ topk_idx,
                                                                   float* __restrict__ topk_w, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int n = *flagged_count;
  if (!dcheck(n <= T, status)) return;
  const int lane = threadIdx.x & 31;
  for (int i = blockIdx.x * 8 + (threadIdx.x >> 5); i < n; i += gridDim.x * 8) {
    float l[kMaxPerLane];
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) l[j] = 0.f;
    for (int z = 0; z < splits; ++z) {  // eight independent loads per part, summed in part order
      const float* row = part + (static_cast<size_t>(z) * n + i) * E;
      float v[kMaxPerLane];
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) v[j] = (lane + 32 * j < E) ? row[lane + 32 * j] : 0.f;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) l[j] += v[j];
    }
    float sv[kMaxPerLane];
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) sv[j] = (lane + 32 * j < E) ? sigmoid(l[j]) : 0.f;
    if (!dcheck(flagged[i] >= 0 && flagged[i] < T, status)) continue;
    warp_select(sv, bias, lane, flagged[i], E, G, Gk, K, scale, topk_idx, topk_w, status);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 router_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// bf16 matrix [outer][inner], boxes of box_inner x box_outer with the given
// swizzle; rows past the end read as zero.
int encode_router_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto fn = router_encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

// fp32 matrix [outer][inner] (row stride `stride` elements), boxes of
// box_inner x box_outer, no swizzle; rows past the end read as zero.
int encode_f32_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t stride,
                   uint32_t box_inner, uint32_t box_outer) {
  auto fn = router_encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {stride * 4};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

}  // namespace

int router_epad(int E) { return ((E + 15) / 16) * 16; }

namespace {

// CTAs of a tensor-core router cluster: 4, or 2 where a quarter of the
// expert rows would not be whole 8-row swizzle atoms.
int tc_cluster(int E_pad) { return E_pad % 32 == 0 ? 4 : 2; }

// Token tiles of the tensor-core router's grid: whole clusters (tiles past
// the batch read zero tokens and write nothing).
int tc_cluster_tiles(int T) {
  constexpr int kC = 4;
  return ((T + kTcTokens - 1) / kTcTokens + kC - 1) / kC * kC;
}

}  // namespace

// The fp32 recompute works on hidden-dimension parts of whole 32-row chunks,
// and its x slice, W_r ring and partial sums must fit in shared memory.
bool router_uses_tensor_cores(int T, int E, int d) {
  const size_t smem = sizeof(float4) * static_cast<size_t>(d / flag_splits(d)) +
                      sizeof(float) * static_cast<size_t>(kFlagRing) * kFlagRows * E +
                      sizeof(float) * 4 * kFlagTokens * 256 + 1024;
  return T >= kRouterTcMinTokens && router_epad(E) <= 256 && d % (flag_splits(d) * kFlagRows) == 0 &&
         smem <= 232448;
}

// Split of the hidden dimension over CTAs: the largest that keeps all CTAs in
// one wave (one CTA per SM), so small batches still use most SMs.
int router_tc_splits(int T, int d, int num_sms) {
  const int tiles = tc_cluster_tiles(T);
  const int kblocks = d / kTcBK;
  int best = 1;
  for (int s = 1; s <= kTcMaxSplits && s <= kblocks; ++s)
    if (kblocks % s == 0 && tiles * s <= num_sms) best = s;
  return best;
}

// Splits of the hidden dimension the scratch is sized for (the split grows with
// the SM count; 1024 SMs bound every device).
int router_tc_max_splits(int T, int d) { return router_tc_splits(std::max(T, 1), d, 1024); }

namespace {

size_t up256(size_t b) { return (b + 255) & ~size_t(255); }

// Tensor-core router scratch: the split W_r [3][E_pad][d] bf16, the flagged
// tokens [T], the column sums of squares [d/128][E32] and the strips' largest
// column norms [8] fp32.
struct TcScratch {
  uint16_t* w_split;
  int32_t* flagged;
  float* colss;
  float* wn_strip;
  size_t bytes;
};

TcScratch tc_scratch(void* base, int T, int d, int E) {
  const int E_pad = router_epad(E), E32 = (E_pad + 31) / 32 * 32;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t o = 0;
  TcScratch s;
  s.w_split = reinterpret_cast<uint16_t*>(p + o);
  o += up256(sizeof(uint16_t) * 3 * E_pad * static_cast<size_t>(d));
  s.flagged = reinterpret_cast<int32_t*>(p + o);
  o += up256(sizeof(int32_t) * static_cast<size_t>(T));
  s.colss = reinterpret_cast<float*>(p + o);
  o += up256(sizeof(float) * static_cast<size_t>(d / kWsRows) * E32);
  s.wn_strip = reinterpret_cast<float*>(p + o);
  o += 256;
  s.bytes = o;
  return s;
}

}  // namespace

size_t router_tc_scratch_bytes(int T, int d, int E) { return tc_scratch(nullptr, T, d, E).bytes; }

// Tensor-core accumulation error constant of the flag bound (kappa). Measured
// |logit error| / (2^-23 sqrt(d/16) |x_t| |W_r[:, e]|), maximum over a million
// logits per input: 0.047-0.057 for normal activations and router weights
// (also scaled by 3 and 0.7, with 1 % outlier channels at 20x, heavy-tailed,
// and the skewed workload), 0.067 at d = 256, and 0.096 with router columns
// strongly aligned with the tokens (logits up to 12.5, partial sums near
// their Cauchy-Schwarz bound). kappa keeps a factor of 3 above the worst.
constexpr float kTcErrKappa = 0.3f;

cudaError_t launch_router_tc(const uint16_t* x, const float* w_r, void* scratch, float* part, int32_t* flagged_count,
                             int32_t* hdr_ticket, int T, int d, int E, int n_groups, int topk_groups, int top_k,
                             float routed_scale, const float* sel_bias, int32_t* topk_idx, float* topk_w,
                             int32_t* status, int32_t* timeout_where, long long wait_spins, int num_sms,
                             cudaStream_t stream) {
  const int E_pad = router_epad(E);
  const TcScratch sc = tc_scratch(scratch, T, d, E);
  const dim3 split_grid(d / kWsRows, (E_pad + 31) / 32);
  cudaError_t err = launch_pdl(wr_split_kernel, split_grid, dim3(256), 0, stream, w_r, d, E, E_pad, sc.w_split, sc.colss,
                               sc.wn_strip, hdr_ticket, flagged_count);
  if (err != cudaSuccess) return err;
  CUtensorMap tmX, tmW;
  const int cluster = tc_cluster(E_pad);
  if (encode_router_map(&tmX, x, d, T, kTcBK, kTcTokens, CU_TENSOR_MAP_SWIZZLE_64B) ||
      encode_router_map(&tmW, sc.w_split, d, 3ull * E_pad, kTcBK, static_cast<uint32_t>(E_pad / cluster),
                        CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int splits = std::min(router_tc_splits(T, d, num_sms), router_tc_max_splits(T, d));
  TcArgs a;
  a.T = T;
  a.d = d;
  a.E = E;
  a.E_pad = E_pad;
  a.kb_per_split = d / kTcBK / splits;
  a.part = part;
  a.status = status;
  a.timeout_where = timeout_where;
  a.wait_spins = wait_spins;
  a.stage_bytes = ((kTcTokens * kTcBK * 2 + 3 * E_pad * kTcBK * 2) + 1023u) & ~1023u;
  a.tmem_cols = 32;
  while (a.tmem_cols < static_cast<uint32_t>(2 * E_pad)) a.tmem_cols <<= 1;
  a.cluster = cluster;
  const size_t smem = 1024 + static_cast<size_t>(kTcStages) * a.stage_bytes;
  err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tc_cluster_tiles(T), splits);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, router_tc_kernel, tmX, tmW, a);
  }
  if (err != cudaSuccess) return err;
  const float err_coef = kTcErrKappa * 0x1p-23f * sqrtf(static_cast<float>(d) / 16.0f);
  err = launch_pdl(router_select_flag_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, part, splits, T, E, n_groups,
                   topk_groups, top_k, routed_scale, sel_bias, x, d, sc.wn_strip, static_cast<int>(split_grid.y),
                   err_coef, topk_idx, topk_w, sc.flagged, flagged_count, status);
  if (err != cudaSuccess) return err;
  // the tensor-core partials were consumed by the selection: reuse `part` for the recompute
  const int fsplits = flag_splits(d);
  const size_t xs_bytes = sizeof(float4) * static_cast<size_t>(d / fsplits) +
                          sizeof(float) * static_cast<size_t>(kFlagRing) * kFlagRows * E;
  err = cudaFuncSetAttribute(router_flagged_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(xs_bytes));
  if (err != cudaSuccess) return err;
  err = launch_pdl(router_flagged_logits_kernel, dim3(num_sms), dim3(kFlagThreads), xs_bytes, stream, x, w_r, T, d,
                   E, sc.flagged, flagged_count, part, fsplits, status, timeout_where, wait_spins);
  if (err != cudaSuccess) return err;
  return launch_pdl(router_flagged_select_kernel, dim3(num_sms), dim3(256), 0, stream, part, fsplits, T, E, n_groups,
                    topk_groups, top_k, routed_scale, sel_bias, sc.flagged, flagged_count, topk_idx, topk_w, status);
}

static_assert(sizeof(WsHeader::route_ticket) == sizeof(int32_t) * kRouteTickets, "ticket array size");

bool router_simt_selects(int T) { return ((T + kRsTokens - 1) / kRsTokens) * kRsCluster <= kRouteTickets; }

size_t router_simt_scratch_bytes(int d, int E) {
  return E % 4 ? sizeof(float) * static_cast<size_t>(d) * ((E + 3) & ~3) : 0;
}

cudaError_t launch_router_simt(const uint16_t* x, const float* w_r, void* scratch, float* logits, int32_t* ticket,
                               int T, int d, int E, int n_groups, int topk_groups, int top_k, float routed_scale,
                               const float* sel_bias, int32_t* topk_idx, float* topk_w, int32_t* status,
                               int32_t* timeout_where, long long wait_spins, int num_sms, cudaStream_t stream) {
  const float* w = w_r;
  int E4 = E;
  cudaError_t err;
  if (E % 4) {
    E4 = (E + 3) & ~3;
    float* wp = static_cast<float*>(scratch);
    err = launch_pdl(wr_pad_kernel, dim3(num_sms), dim3(256), 0, stream, w_r, d, E, E4, wp);
    if (err != cudaSuccess) return err;
    w = wp;
  }
  CUtensorMap tmX, tmW;
  if (encode_router_map(&tmX, x, d, T, kRsBK, kRsTokens, CU_TENSOR_MAP_SWIZZLE_128B) ||
      encode_f32_map(&tmW, w, E4, d, E4, kRsExperts, kRsBK))
    return cudaErrorInvalidValue;
  const bool selects = router_simt_selects(T);
  RsArgs a;
  a.T = T;
  a.d = d;
  a.E = E;
  a.G = n_groups;
  a.Gk = topk_groups;
  a.K = top_k;
  a.scale = routed_scale;
  a.bias = sel_bias;
  a.logits = logits;
  a.ticket = selects ? ticket : nullptr;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.status = status;
  a.timeout_where = timeout_where;
  a.wait_spins = wait_spins;
  const size_t smem = 1024 + static_cast<size_t>(kRsStages) * kRsStageBytes;
  err = cudaFuncSetAttribute(router_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid((T + kRsTokens - 1) / kRsTokens, (E + kRsExperts - 1) / kRsExperts, kRsCluster);
  err = launch_pdl(router_simt_kernel, grid, dim3(kRsThreads), smem, stream, tmX, tmW, a);
  if (err != cudaSuccess || selects) return err;
  return launch_pdl(router_select_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, logits, T, E, n_groups,
                    topk_groups, top_k, routed_scale, sel_bias, topk_idx, topk_w, status);
}

}  // namespace beammoe
