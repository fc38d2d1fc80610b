// Router of the Beam MoE block (release article, section "Mixture of
// Experts": sigmoid scores over all experts, groups ranked by the sum of
// their two best scores, the best groups kept, the top experts inside them
// chosen, weights normalised then scaled by 2.5; FP32 router per section
// "Residual stream").
//
// Small batches (decode):
//  router_logits_kernel  FP32 SIMT GEMM, logits = x . W_r, with a split over
//                        the hidden dimension so the whole GPU streams W_r.
//  split_reduce_kernel   sums the split partials of each logit in a fixed
//                        order (four interleaved chains, then pairwise), in
//                        place into split 0.
//  router_select_kernel  one warp per token: sigmoid, group top-2 sums, top
//                        groups, top experts, normalisation.
// Large batches (prefill):
//  wr_split_kernel       W_r (fp32, [d][E]) -> three bf16 matrices hi, mid,
//                        lo ([E_pad][d], K-contiguous) with hi + mid + lo = W_r
//                        (8 + 8 + 8 significant bits cover fp32's 24), and the
//                        largest column norm of W_r (a fixed-order reduction).
//  router_tc_kernel      per 128 tokens and one range of the hidden dimension:
//                        partial logits x.hi + x.mid + x.lo on the tcgen05
//                        tensor cores (x is exact in bf16, so every product is
//                        exact in fp32).
//  router_select_flag_kernel  one warp per token: partials summed, sigmoid,
//                        group-limited selection and the two decision margins.
//                        The tensor cores' fp32 accumulation is coarser than
//                        FFMA, so a decision is kept only where every margin
//                        exceeds a bound on the logit error that scales with
//                        the token: kappa * 2^-23 * sqrt(d/16) * |x_t| *
//                        max_e |W_r[:, e]| (every partial sum of x_t . W_r[:, e]
//                        is at most |x_t| |W_r[:, e]| by Cauchy-Schwarz, and
//                        d/16 MMA steps each round once; kappa is set from
//                        measured errors with a wide margin). |x_t| comes from
//                        the tensor-core kernel's epilogue warps, the column
//                        norms of W_r from wr_split_kernel. Elsewhere:
//  router_flagged_logits_kernel, router_flagged_select_kernel: tokens with a
//                        narrow margin get all logits in fp32 FFMA and the
//                        full warp selection.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int RT = 64;   // tokens per block
constexpr int RE = 128;  // experts per block
constexpr int RK = 32;   // hidden elements per smem stage

__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ wr,
                                                            float* __restrict__ part, int T, int d, int E,
                                                            int k_per_split) {
  __shared__ __align__(16) float xs[RK][RT + 4];  // xs[k][t]
  __shared__ __align__(16) float ws[RK][RE];      // ws[k][e]
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int e0 = blockIdx.x * RE, t0 = blockIdx.y * RT;
  const int kbeg = blockIdx.z * k_per_split, kend = kbeg + k_per_split;
  const bool vec_w = (E & 3) == 0;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = kbeg; k0 < kend; k0 += RK) {
    {
      const int r = tid >> 2, kc = (tid & 3) * 8, t = t0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + k0 + kc);
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[kc + i][r] = bf16_bits_to_float(h[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = tid + 256 * i, kk = q >> 5, ec = (q & 31) * 4, e = e0 + ec;
      const float* src = wr + static_cast<size_t>(k0 + kk) * E + e;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (vec_w && e + 3 < E) {
        v = *reinterpret_cast<const float4*>(src);
      } else {
        if (e + 0 < E) v.x = src[0];
        if (e + 1 < E) v.y = src[1];
        if (e + 2 < E) v.z = src[2];
        if (e + 3 < E) v.w = src[3];
      }
      *reinterpret_cast<float4*>(&ws[kk][ec]) = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&ws[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&ws[kk][tx * 8 + 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* dst = part + static_cast<size_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + tx * 8 + j;
      if (e < E) dst[static_cast<size_t>(t) * E + e] = acc[i][j];
    }
  }
}

// part[0][t][e] = sum over s of part[s][t][e] in a fixed order: four chains
// over s = 0,4,8,.. / 1,5,.. / 2,6,.. / 3,7,.. (independent loads in flight),
// then (c0 + c1) + (c2 + c3).
__global__ void __launch_bounds__(256) split_reduce_kernel(float* __restrict__ part, int splits, int64_t n) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
  int sp = 0;
  for (; sp + 4 <= splits; sp += 4) {
    c0 += part[static_cast<size_t>(sp) * n + i];
    c1 += part[static_cast<size_t>(sp + 1) * n + i];
    c2 += part[static_cast<size_t>(sp + 2) * n + i];
    c3 += part[static_cast<size_t>(sp + 3) * n + i];
  }
  for (; sp < splits; ++sp) c0 += part[static_cast<size_t>(sp) * n + i];
  part[i] = (c0 + c1) + (c2 + c3);
}

// (value, index) order of the selection: larger value first, ties to the
// lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

constexpr int kMaxPerLane = 8;  // E <= 256

// Group-limited selection of one token by one warp. Lane l holds the scores
// of experts l, l+32, l+64, ... in s[]; `bias` ([E] fp32, nullable) is the
// per-expert selection bias of DeepSeek-V3-style balancing: groups and
// experts are chosen on s + bias, the weights use s. Writes the token's K
// expert ids (slot order: descending selection score, ties to the lower id)
// and weights. Returns, in every lane, the decision margins (on selection
// scores): x = worst kept group score - best dropped one; y = the smaller of
// (worst chosen score - best unchosen candidate) and the gaps between
// consecutive slots.
__device__ float2 warp_select(const float (&s_in)[kMaxPerLane], const float* __restrict__ bias, int lane, int t,
                              int E, int G, int Gk, int K, float scale, int32_t* __restrict__ topk_idx,
                              float* __restrict__ topk_w, int32_t* status) {
  const int gsz = E / G;
  constexpr float kMasked = -1.0f;  // below every sigmoid score
  float s[kMaxPerLane];             // selection scores
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = (bias && e < E) ? s_in[i] + bias[e] : s_in[i];
  }
  int grp[kMaxPerLane];             // group of each of this lane's experts (E = none)
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    grp[i] = (e < E) ? e / gsz : 64;
  }

  // group score: sum of the two largest scores of the group (lane g keeps group g's)
  float my_gs = kMasked;
  if (gsz == 32) {
    // element i of every lane is group i: all groups reduce side by side
    float m1[kMaxPerLane], m2[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      m1[i] = s[i];
      m2[i] = kMasked;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const float o1 = __shfl_xor_sync(0xffffffffu, m1[i], off);
        const float o2 = __shfl_xor_sync(0xffffffffu, m2[i], off);
        if (o1 > m1[i]) {
          m2[i] = fmaxf(m1[i], o2);
          m1[i] = o1;
        } else {
          m2[i] = fmaxf(m2[i], o1);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (lane == i && i < G) my_gs = m1[i] + m2[i];
  }
  for (int g = 0; g < G && gsz != 32; ++g) {
    float m1 = kMasked, m2 = kMasked;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      if (grp[i] == g) {
        if (s[i] > m1) {
          m2 = m1;
          m1 = s[i];
        } else if (s[i] > m2) {
          m2 = s[i];
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, m1, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
      if (o1 > m1) {
        m2 = fmaxf(m1, o2);
        m1 = o1;
      } else {
        m2 = fmaxf(m2, o1);
      }
    }
    if (lane == g) my_gs = (gsz >= 2) ? (m1 + m2) : m1;
  }

  // keep the Gk best groups (ties to the lower group index)
  uint32_t kept = 0;
  float last_kept = 0.f;
  for (int r = 0; r < Gk; ++r) {
    float v = (lane < G && !((kept >> lane) & 1u)) ? my_gs : -2.0f;
    int i = lane;
    warp_argmax(v, i);
    kept |= 1u << i;
    last_kept = v;
  }
  float margin_group = 1.0f, margin = 1.0f;
  {
    float v = (lane < G && !((kept >> lane) & 1u)) ? my_gs : -2.0f;
    int i = lane;
    warp_argmax(v, i);
    if (v > -1.5f) margin_group = last_kept - v;
  }

  // choose the K best experts of the kept groups (ties to the lower index)
  uint32_t taken = 0;  // bit i: this lane's element i is chosen
  float my_s = 0.f;    // slot `lane`: its selection score ...
  float my_w = 0.f;    // ... and its unbiased score (the weight's)
  int my_e = 0;
  float sum = 0.f;     // of unbiased scores
  for (int k = 0; k < K; ++k) {
    float v = -2.0f;
    int idx = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (grp[i] < 32 && ((kept >> grp[i]) & 1u) && !((taken >> i) & 1u) && better(s[i], e, v, idx)) {
        v = s[i];
        idx = e;
      }
    }
    warp_argmax(v, idx);
    float u = 0.f;  // the chosen expert's unbiased score, from the lane that holds it
    if (idx >= E || idx < 0) {  // only possible with NaN scores
      latch_status(status, MOE_DEV_BAD_EXPERT);
      idx = 0;
      v = 0.f;
    } else {
      if ((idx & 31) == lane) taken |= 1u << (idx >> 5);
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (i == (idx >> 5)) u = s_in[i];
      u = __shfl_sync(0xffffffffu, u, idx & 31);
    }
    sum += u;
    if (lane == k) {
      my_s = v;
      my_w = u;
      my_e = idx;
    }
  }
  {
    float v = -2.0f;
    int idx = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (grp[i] < 32 && ((kept >> grp[i]) & 1u) && !((taken >> i) & 1u) && better(s[i], e, v, idx)) {
        v = s[i];
        idx = e;
      }
    }
    warp_argmax(v, idx);
    const float last_s = __shfl_sync(0xffffffffu, my_s, K - 1);
    if (v > -1.5f) margin = fminf(margin, last_s - v);
    // gaps between consecutive slots: the slot order is a decision too
    const float next_s = __shfl_down_sync(0xffffffffu, my_s, 1);
    float gap = (lane + 1 < K) ? my_s - next_s : 1.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gap = fminf(gap, __shfl_xor_sync(0xffffffffu, gap, off));
    margin = fminf(margin, gap);
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
    s[i] = (e < E) ? 1.0f / (1.0f + expf(-logits[static_cast<size_t>(t) * E + e])) : -1.0f;
  }
  warp_select(s, bias, lane, t, E, G, Gk, K, scale, topk_idx, topk_w, status);
}

// ---------------------------------------------------------------- tensor-core path

constexpr int kTcTokens = 128;  // tokens per CTA (MMA M)
constexpr int kTcBK = 64;       // hidden elements per pipeline stage
constexpr int kTcStages = 2;
constexpr int kTcMaxSplits = 16;
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint64_t kTcDrainNs = 1000000000ull;

// out[s][e][k] = bf16 split s of W_r[k][e] (rows e >= E are zero). Also
// resets the flagged-token count, and finds the largest column norm of W_r in
// a fixed order: every block writes the sums of squares of its 32 x 32 tile's
// columns to colss[k block][e]; the last block to finish a 32-expert strip
// (counted in ticket[strip], which it returns to 0) adds them up in k order
// and writes the strip's largest norm to wn_strip[strip].
__global__ void __launch_bounds__(256) wr_split_kernel(const float* __restrict__ wr, int d, int E, int E_pad,
                                                       uint16_t* __restrict__ out, float* __restrict__ colss,
                                                       float* __restrict__ wn_strip, int32_t* __restrict__ ticket,
                                                       int32_t* __restrict__ flagged_count) {
  __shared__ float tile[32][33];
  __shared__ int is_last;
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *flagged_count = 0;
  const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int E32 = gridDim.y * 32;  // row stride of colss
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + tx;
    tile[i][tx] = (e < E) ? wr[static_cast<size_t>(k0 + i) * E + e] : 0.f;
  }
  __syncthreads();
  if (ty == 0) {
    float ss = 0.f;
#pragma unroll 8
    for (int k = 0; k < 32; ++k) ss = fmaf(tile[k][tx], tile[k][tx], ss);
    colss[static_cast<size_t>(blockIdx.x) * E32 + e0 + tx] = ss;
  }
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, k = k0 + tx;
    if (e >= E_pad) continue;
    const float w = tile[tx][i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    const size_t o = static_cast<size_t>(e) * d + k;
    const size_t plane = static_cast<size_t>(E_pad) * d;
    out[o] = __bfloat16_as_ushort(hi);
    out[plane + o] = __bfloat16_as_ushort(mid);
    out[2 * plane + o] = __bfloat16_as_ushort(lo);
  }
  __threadfence();  // this block's column sums are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&ticket[blockIdx.y], 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (is_last && ty == 0) {
    float ss = 0.f;
    for (int kx = 0; kx < static_cast<int>(gridDim.x); ++kx) ss += __ldcg(colss + static_cast<size_t>(kx) * E32 + e0 + tx);
    float nrm = sqrtf(ss);
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
  const uint16_t* x; // [T][d] (read by the epilogue warps for the token norms)
  float* xss;        // [splits][T] partial sums of squares of x over each CTA's hidden range
  int32_t* status;
  int32_t* timeout_where;
  long long wait_spins;
  uint32_t stage_bytes;
  uint32_t tmem_cols;
};

__device__ __forceinline__ void tc_fail(const TcArgs& a, volatile int* abort, int where) {
  latch_status(a.status, MOE_DEV_TIMEOUT);
  if (a.timeout_where) atomicCAS(a.timeout_where, 0, where);
  *abort = 1;
}

// Partial logits of 128 tokens x E_pad experts over one range of the hidden
// dimension: hi products accumulate in D1 (TMEM columns [0, E_pad)), the small
// mid and lo products in D2 ([E_pad, 2 E_pad)), so they keep their bits.
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
  constexpr uint32_t kXTile = kTcTokens * kTcBK * 2;                  // 16 KB

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
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
  __syncthreads();
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
        for (int sp = 0; sp < 3; ++sp)
          tma_load_2d(st + kXTile + sp * wtile, &tmW, kb * kTcBK, sp * a.E_pad, &full_bar[stage]);
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
          const uint64_t adesc = sdesc_kmajor_sw128(sx + k * 32);
          const uint32_t first = ((kb - kb0) | k) != 0 ? 1u : 0u;
          mma_bf16_ss(tmem_base, adesc, sdesc_kmajor_sw128(sx + kXTile + k * 32), idesc, first);
          mma_bf16_ss(tmem_base + a.E_pad, adesc, sdesc_kmajor_sw128(sx + kXTile + wtile + k * 32), idesc, first);
          mma_bf16_ss(tmem_base + a.E_pad, adesc, sdesc_kmajor_sw128(sx + kXTile + 2 * wtile + k * 32), idesc, 1u);
        }
        mma_commit(&empty_bar[stage]);
        if (++stage == kTcStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(&accf_bar);
    }
    __syncwarp();
  } else {
    // epilogue: thread r owns token t0 + r (TMEM lane r). While the MMAs run it
    // sums the squares of its token's x over this CTA's hidden range (the
    // token norm of the flag bound); then the partial logits go to global.
    const int q = warp & 3, r = q * 32 + lane;
    const int t = t0 + r;
    if (t < a.T) {
      const int k0 = kb0 * kTcBK, n8 = (kb1 - kb0) * kTcBK / 8;
      const uint4* row = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.d + k0);
      float ss = 0.f;
      for (int i = 0; i < n8; ++i) {
        const uint4 v = __ldg(row + i);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(w4[j] << 16), hi = __uint_as_float(w4[j] & 0xFFFF0000u);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
      a.xss[static_cast<size_t>(blockIdx.y) * a.T + t] = ss;
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&accf_bar, 0, a.wait_spins, kTcWaitNs, abort));
    if (ok) {
      tc_fence_after();
      float* dst = a.part + (static_cast<size_t>(blockIdx.y) * a.T + t) * a.E;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      for (int c = 0; c < a.E_pad; c += 16) {
        uint32_t v[16], v2[16];
        tmem_ld_32x32b_x16(tb + c, v);
        tmem_ld_32x32b_x16(tb + a.E_pad + c, v2);
        tmem_ld_wait();
        if (t < a.T) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < a.E) dst[c + j] = __uint_as_float(v[j]) + __uint_as_float(v2[j]);
        }
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
                                                                 const float* __restrict__ xss,
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
  float xs = 0.f;
  for (int sp = 0; sp < splits; ++sp) {  // eight independent loads per split, summed in split order
    const float* row = part + (static_cast<size_t>(sp) * T + t) * E;
    float v[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) v[i] = (lane + 32 * i < E) ? row[lane + 32 * i] : 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) l[i] += v[i];
    xs += xss[static_cast<size_t>(sp) * T + t];
  }
  float wn = 0.f;
  for (int i = 0; i < n_strips; ++i) wn = fmaxf(wn, wn_strip[i]);
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = (e < E) ? 1.0f / (1.0f + expf(-l[i])) : -1.0f;
  }
  const float2 margin = warp_select(s, bias, lane, t, E, G, Gk, K, scale, topk_idx, topk_w, status);
  const float e_s = 0.25f * err_coef * sqrtf(xs) * wn;
  const bool narrow = !(margin.x >= 4.f * e_s && margin.y >= 2.f * e_s);  // NaN margins are narrow too
  if (lane == 0 && narrow) flagged[atomicAdd(flagged_count, 1)] = t;
}

// Flagged tokens: every logit as an fp32 FFMA dot product. Work items are
// (group of up to kFlagTokens flagged tokens, one of `splits` parts of the
// hidden dimension: 8, or 4 where d is not a multiple of 8 x 32), taken
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
    float sv[kMaxPerLane];
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      const int e = lane + 32 * j;
      sv[j] = -1.0f;
      if (e < E) {
        float l = 0.f;
        for (int z = 0; z < splits; ++z) l += part[(static_cast<size_t>(z) * n + i) * E + e];
        sv[j] = 1.0f / (1.0f + expf(-l));
      }
    }
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

int encode_router_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = router_encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

}  // namespace

int router_epad(int E) { return ((E + 15) / 16) * 16; }

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
  const int tiles = (T + kTcTokens - 1) / kTcTokens;
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
// tokens [T], the column sums of squares [d/32][E32] and the strips' largest
// column norms [8] fp32, and the token sums of squares [splits][T] fp32.
struct TcScratch {
  uint16_t* w_split;
  int32_t* flagged;
  float* colss;
  float* wn_strip;
  float* xss;
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
  o += up256(sizeof(float) * static_cast<size_t>(d / 32) * E32);
  s.wn_strip = reinterpret_cast<float*>(p + o);
  o += 256;
  s.xss = reinterpret_cast<float*>(p + o);
  o += up256(sizeof(float) * static_cast<size_t>(router_tc_max_splits(T, d)) * T);
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
  const dim3 split_grid(d / 32, (E_pad + 31) / 32);
  cudaError_t err = launch_pdl(wr_split_kernel, split_grid, dim3(256), 0, stream, w_r, d, E, E_pad, sc.w_split, sc.colss,
                               sc.wn_strip, hdr_ticket, flagged_count);
  if (err != cudaSuccess) return err;
  CUtensorMap tmX, tmW;
  if (encode_router_map(&tmX, x, d, T, kTcTokens) || encode_router_map(&tmW, sc.w_split, d, 3ull * E_pad, E_pad))
    return cudaErrorInvalidValue;
  const int splits = std::min(router_tc_splits(T, d, num_sms), router_tc_max_splits(T, d));
  TcArgs a;
  a.T = T;
  a.d = d;
  a.E = E;
  a.E_pad = E_pad;
  a.kb_per_split = d / kTcBK / splits;
  a.part = part;
  a.x = x;
  a.xss = sc.xss;
  a.status = status;
  a.timeout_where = timeout_where;
  a.wait_spins = wait_spins;
  a.stage_bytes = ((kTcTokens * kTcBK * 2 + 3 * E_pad * kTcBK * 2) + 1023u) & ~1023u;
  a.tmem_cols = 32;
  while (a.tmem_cols < static_cast<uint32_t>(2 * E_pad)) a.tmem_cols <<= 1;
  const size_t smem = 1024 + static_cast<size_t>(kTcStages) * a.stage_bytes;
  err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  err = launch_pdl(router_tc_kernel, dim3((T + kTcTokens - 1) / kTcTokens, splits), dim3(192), smem, stream, tmX, tmW,
                   a);
  if (err != cudaSuccess) return err;
  const float err_coef = kTcErrKappa * 0x1p-23f * sqrtf(static_cast<float>(d) / 16.0f);
  err = launch_pdl(router_select_flag_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, part, splits, T, E, n_groups,
                   topk_groups, top_k, routed_scale, sel_bias, sc.xss, sc.wn_strip, static_cast<int>(split_grid.y),
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

// Smallest split of the hidden dimension (into >= 64-element slices) that
// gives at least one block per SM.
int router_splits(int T, int d, int E, int num_sms) {
  const int tiles = ((T + RT - 1) / RT) * ((E + RE - 1) / RE);
  const int target = (num_sms + tiles - 1) / tiles;
  const int chunks = d / RK;
  int best = 1;
  for (int s = 1; s <= chunks; ++s) {
    if (chunks % s || d / s < 64) continue;
    best = s;
    if (s >= target) break;
  }
  return best;
}

cudaError_t launch_router_logits(const uint16_t* x, const float* w_r, float* partial, int T, int d, int E,
                                 int splits, cudaStream_t stream) {
  const dim3 grid((E + RE - 1) / RE, (T + RT - 1) / RT, splits);
  return launch_pdl(router_logits_kernel, grid, dim3(256), 0, stream, x, w_r, partial, T, d, E, d / splits);
}

cudaError_t launch_router_select(float* partial, int splits, int T, int E, int n_groups, int topk_groups,
                                 int top_k, float routed_scale, const float* sel_bias, int32_t* topk_idx,
                                 float* topk_w, int32_t* status, cudaStream_t stream) {
  if (splits > 1) {
    const int64_t n = static_cast<int64_t>(T) * E;
    const cudaError_t err = launch_pdl(split_reduce_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                                       stream, partial, splits, n);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(router_select_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, partial, T, E, n_groups,
                    topk_groups, top_k, routed_scale, sel_bias, topk_idx, topk_w, status);
}

}  // namespace beammoe
