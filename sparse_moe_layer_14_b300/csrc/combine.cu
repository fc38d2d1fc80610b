// Combine of the Beam MoE block (release article, section "Mixture of
// Experts": expert outputs summed with the normalised router weights, scaled
// by 2.5 -- the scale is already inside topk_w -- and no shared expert).
//
// out[t][c] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*K+k]][c] ), the sum
// in FP32 in slot order (deterministic, no atomics) over the FP32 expert
// outputs. Each thread owns four consecutive columns: one 16-byte load of
// every slot's row (all K loads issued before the first use), one 8-byte
// store. HBM-bound: K*d*4 bytes read and d*2 written per token.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 8;  // slots loaded in flight per pass (Beam's top-8 in one pass)

// Weighted sum over one token's slots of four consecutive columns c..c+3 (FP32, slot
// order); a row index outside [0, R) is skipped and latched once (by `latcher`).
__device__ __forceinline__ float4 combine4(const float* __restrict__ y, const int32_t* __restrict__ inv_row,
                                           const float* __restrict__ topk_w, int t, int c, int d, int K, int64_t R,
                                           bool load, bool latcher, int32_t* status) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < K; k0 += kMaxK) {
    const int nk = min(kMaxK, K - k0);
    float4 v[kMaxK];
    float w[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      w[k] = 0.f;
      if (k < nk) {
        const int r = inv_row[static_cast<size_t>(t) * K + k0 + k];
        if (r < 0 || r >= R) {
          if (latcher) latch_status(status, MOE_DEV_BAD_ROW);
        } else if (load) {
          w[k] = topk_w[static_cast<size_t>(t) * K + k0 + k];
          v[k] = *reinterpret_cast<const float4*>(y + static_cast<size_t>(r) * d + c);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {  // slot order
      if (k < nk) {
        acc.x = fmaf(w[k], v[k].x, acc.x);
        acc.y = fmaf(w[k], v[k].y, acc.y);
        acc.z = fmaf(w[k], v[k].z, acc.z);
        acc.w = fmaf(w[k], v[k].w, acc.w);
      }
    }
  }
  return acc;
}

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

__global__ void __launch_bounds__(kThreads, 8) combine_kernel(const float* __restrict__ y,
                                                           const int32_t* __restrict__ inv_row,
                                                           const float* __restrict__ topk_w,
                                                           uint16_t* __restrict__ out, int T, int d, int K,
                                                           int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kThreads + threadIdx.x) * 4;
  if (c >= d) return;
  const float4 acc = combine4(y, inv_row, topk_w, t, c, d, K, static_cast<int64_t>(T) * K, true, c == 0, status);
  *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d + c) = pack4_bf16(acc.x, acc.y, acc.z, acc.w);
}

// Combine fused with the post-norm and the depth-scaled residual addition
// (release article, section "Residual stream": every sublayer is normalised
// after, and at step k the stream keeps weight sqrt((k-1)/k) and takes the
// sublayer output with weight 1/sqrt(k); the norms in FP32). The blocks of
// one token's row form a thread-block cluster (1024 columns per block: a
// cluster of d/1024 <= 8): each block combines its columns like combine_kernel
// (all K loads in flight, FP32 sum in slot order), publishes its partial sum
// of squares in shared memory, and after a cluster barrier every block reads
// the others' partials through distributed shared memory for
//   r = sqrt(mean(out^2) + eps),
// then resid[t][c] = bf16( keep * resid[t][c] + add * out[c] / r * gain[c] ),
// in place. One read of the K rows and of the residual row, one write.
constexpr int kResThreads = 256;
constexpr int kResColsPerBlock = kResThreads * 4;  // 1024
constexpr int kResMaxCluster = 8;

__global__ void __launch_bounds__(kResThreads, 4) combine_residual_kernel(
    const float* __restrict__ y, const int32_t* __restrict__ inv_row, const float* __restrict__ topk_w,
    const uint16_t* __restrict__ gain, float eps, float keep, float add, uint16_t* __restrict__ resid, int T, int d,
    int K, int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float warp_ss[kResThreads / 32];
  __shared__ float block_ss;
  __shared__ float inv_r;
  const int nb = static_cast<int>(cluster.num_blocks());  // column blocks of the row
  const int t = static_cast<int>(blockIdx.x) / nb;
  const int cb = static_cast<int>(cluster.block_rank());
  const int c = cb * kResColsPerBlock + threadIdx.x * 4;
  const bool active = c < d;  // no early return: every thread meets the cluster barrier
  const float4 acc = combine4(y, inv_row, topk_w, t, c, d, K, static_cast<int64_t>(T) * K, active,
                              threadIdx.x == 0 && cb == 0, status);
  uint2 h = make_uint2(0, 0), g = make_uint2(0, 0);
  if (active) {  // in flight across the reduction
    h = *reinterpret_cast<const uint2*>(resid + static_cast<size_t>(t) * d + c);
    g = *reinterpret_cast<const uint2*>(gain + c);
  }
  float ss = acc.x * acc.x;
  ss = fmaf(acc.y, acc.y, ss);
  ss = fmaf(acc.z, acc.z, ss);
  ss = fmaf(acc.w, acc.w, ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int i = 0; i < kResThreads / 32; ++i) b += warp_ss[i];
    block_ss = b;
  }
  cluster.sync();  // every block's partial is published
  if (threadIdx.x < 32) {
    // lane j fetches block j's partial; lane 0 adds them in rank order (the same sum in every block)
    const float part = threadIdx.x < nb ? *cluster.map_shared_rank(&block_ss, static_cast<int>(threadIdx.x)) : 0.f;
    float tot = 0.f;
    for (int j = 0; j < nb; ++j) tot += __shfl_sync(0xffffffffu, part, j);
    if (threadIdx.x == 0) inv_r = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  }
  // done reading the other blocks' shared memory (release: the reads above come first); the
  // matching wait is at the end, so its latency hides behind the stores
  asm volatile("barrier.cluster.arrive.aligned;" ::: "memory");
  __syncthreads();
  const float ir = inv_r;
  if (active) {
    const float o[4] = {acc.x, acc.y, acc.z, acc.w};
    const uint32_t hv[2] = {h.x, h.y}, gv[2] = {g.x, g.y};
    float r[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float n0 = o[2 * i] * ir * __uint_as_float(gv[i] << 16);
      const float n1 = o[2 * i + 1] * ir * __uint_as_float(gv[i] & 0xFFFF0000u);
      r[2 * i] = fmaf(keep, __uint_as_float(hv[i] << 16), add * n0);
      r[2 * i + 1] = fmaf(keep, __uint_as_float(hv[i] & 0xFFFF0000u), add * n1);
    }
    *reinterpret_cast<uint2*>(resid + static_cast<size_t>(t) * d + c) = pack4_bf16(r[0], r[1], r[2], r[3]);
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // no block leaves while another may still read it
}

}  // namespace

cudaError_t launch_combine_residual(const float* y_perm, const int32_t* inv_row, const float* topk_w,
                                    const uint16_t* gain, float eps, int step, uint16_t* resid, int T, int d,
                                    int top_k, int32_t* status, cudaStream_t stream) {
  const int nb = (d + kResColsPerBlock - 1) / kResColsPerBlock;
  if (nb > kResMaxCluster) return cudaErrorInvalidValue;  // d > 8192
  const float keep = static_cast<float>(sqrt(static_cast<double>(step - 1) / step));
  const float add = static_cast<float>(1.0 / sqrt(static_cast<double>(step)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(T) * nb));
  cfg.blockDim = dim3(kResThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nb;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, combine_residual_kernel, y_perm, inv_row, topk_w, gain, eps, keep, add, resid, T, d,
                            top_k, status);
}

cudaError_t launch_combine(const float* y_perm, const int32_t* inv_row, const float* topk_w, uint16_t* out,
                           int T, int d, int top_k, int32_t* status, cudaStream_t stream) {
  const dim3 grid(T, (d / 4 + kThreads - 1) / kThreads);
  return launch_pdl(combine_kernel, grid, dim3(kThreads), 0, stream, y_perm, inv_row, topk_w, out, T, d, top_k, status);
}

}  // namespace beammoe
