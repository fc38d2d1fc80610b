// Router of the Beam MoE block (release article, section "Mixture of
// Experts": sigmoid scores over all experts, groups ranked by the sum of
// their two best scores, the best groups kept, the top experts inside them
// chosen, weights normalised then scaled by 2.5; FP32 router per section
// "Residual stream").
//
// Kernels:
//  router_logits_kernel  FP32 SIMT GEMM, logits = x . W_r, with a split over
//                        the hidden dimension when the batch is small so the
//                        whole GPU streams W_r (decode batches).
//  split_reduce_kernel   (split batches only) sums the split partials of each
//                        logit in a fixed order, in place into split 0.
//  router_select_kernel  one warp per token: sigmoid, group top-2 sums, top
//                        groups, top experts, normalisation.
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

// part[0][t][e] = sum over s of part[s][t][e], s ascending.
__global__ void __launch_bounds__(256) split_reduce_kernel(float* __restrict__ part, int splits, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float l = part[i];
  for (int sp = 1; sp < splits; ++sp) l += part[static_cast<size_t>(sp) * n + i];
  part[i] = l;
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

__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits, int T,
                                                            int E, int G, int Gk, int K, float scale,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ topk_w, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int gsz = E / G;
  constexpr float kMasked = -1.0f;  // below every sigmoid score

  float s[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    s[i] = kMasked;
    if (e < E) s[i] = 1.0f / (1.0f + expf(-logits[static_cast<size_t>(t) * E + e]));
  }

  // group score: sum of the two largest scores of the group (lane g keeps group g's)
  float my_gs = kMasked;
  for (int g = 0; g < G; ++g) {
    float m1 = kMasked, m2 = kMasked;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && e / gsz == g) {
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
  for (int r = 0; r < Gk; ++r) {
    float v = (lane < G && !((kept >> lane) & 1u)) ? my_gs : -2.0f;
    int i = lane;
    warp_argmax(v, i);
    kept |= 1u << i;
  }

  // choose the K best experts of the kept groups (ties to the lower index)
  uint32_t taken = 0;  // bit i: this lane's element i is chosen
  float my_s = 0.f;
  int my_e = 0;
  float sum = 0.f;
  for (int k = 0; k < K; ++k) {
    float v = -2.0f;
    int idx = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && ((kept >> (e / gsz)) & 1u) && !((taken >> i) & 1u) && better(s[i], e, v, idx)) {
        v = s[i];
        idx = e;
      }
    }
    warp_argmax(v, idx);
    if (idx >= E || idx < 0) {  // only possible with NaN scores
      latch_status(status, MOE_DEV_BAD_EXPERT);
      idx = 0;
      v = 0.f;
    } else if ((idx & 31) == lane) {
      taken |= 1u << (idx >> 5);
    }
    sum += v;
    if (lane == k) {
      my_s = v;
      my_e = idx;
    }
  }
  if (lane < K) {
    float w = 0.f;
    if (sum > 0.f) {
      w = scale * my_s / sum;
    } else if (lane == 0) {
      latch_status(status, MOE_DEV_ZERO_SUM);
    }
    topk_idx[static_cast<size_t>(t) * K + lane] = my_e;
    topk_w[static_cast<size_t>(t) * K + lane] = w;
  }
}

}  // namespace

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
  dim3 grid((E + RE - 1) / RE, (T + RT - 1) / RT, splits);
  router_logits_kernel<<<grid, 256, 0, stream>>>(x, w_r, partial, T, d, E, d / splits);
  return cudaGetLastError();
}

cudaError_t launch_router_select(float* partial, int splits, int T, int E, int n_groups, int topk_groups,
                                 int top_k, float routed_scale, int32_t* topk_idx, float* topk_w,
                                 int32_t* status, cudaStream_t stream) {
  if (splits > 1) {
    const int64_t n = static_cast<int64_t>(T) * E;
    split_reduce_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(partial, splits, n);
  }
  router_select_kernel<<<(T + 7) / 8, 256, 0, stream>>>(partial, T, E, n_groups, topk_groups, top_k, routed_scale,
                                                         topk_idx, topk_w, status);
  return cudaGetLastError();
}

}  // namespace beammoe
