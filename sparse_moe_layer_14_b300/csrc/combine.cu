// Combine of the Beam MoE block (release article, section "Mixture of
// Experts": expert outputs summed with the normalised router weights, scaled
// by 2.5 -- the scale is already inside topk_w -- and no shared expert).
//
// out[t][c] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*K+k]][c] ), the sum
// in FP32 in slot order (deterministic, no atomics). Each thread owns eight
// consecutive columns: one 16-byte load of every slot's bf16 row (all K loads
// issued before the first use), two 8-byte stores. HBM-bound: K*d*2 bytes
// read and d*2 written per token.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 8;  // slots loaded in flight per pass (Beam's top-8 in one pass)

__device__ __forceinline__ void fma_bf16x2(uint32_t v, float w, float& a, float& b) {
  a = fmaf(w, __uint_as_float(v << 16), a);
  b = fmaf(w, __uint_as_float(v & 0xFFFF0000u), b);
}

__global__ void __launch_bounds__(kThreads, 8) combine_kernel(const uint16_t* __restrict__ y,
                                                           const int32_t* __restrict__ inv_row,
                                                           const float* __restrict__ topk_w,
                                                           uint16_t* __restrict__ out, int T, int d, int K,
                                                           int32_t* status) {
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kThreads + threadIdx.x) * 8;
  if (c >= d) return;
  const int64_t R = static_cast<int64_t>(T) * K;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < K; k0 += kMaxK) {
    const int nk = min(kMaxK, K - k0);
    uint4 v[kMaxK];
    float w[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      w[k] = 0.f;
      if (k < nk) {
        const int r = inv_row[static_cast<size_t>(t) * K + k0 + k];
        if (r < 0 || r >= R) {
          if (c == 0) latch_status(status, MOE_DEV_BAD_ROW);
        } else {
          w[k] = topk_w[static_cast<size_t>(t) * K + k0 + k];
          v[k] = *reinterpret_cast<const uint4*>(y + static_cast<size_t>(r) * d + c);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {  // slot order
      if (k < nk) {
        fma_bf16x2(v[k].x, w[k], acc[0], acc[1]);
        fma_bf16x2(v[k].y, w[k], acc[2], acc[3]);
        fma_bf16x2(v[k].z, w[k], acc[4], acc[5]);
        fma_bf16x2(v[k].w, w[k], acc[6], acc[7]);
      }
    }
  }
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    pk[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint2* o = reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d + c);  // out is 8-byte aligned
  o[0] = make_uint2(pk[0], pk[1]);
  o[1] = make_uint2(pk[2], pk[3]);
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
constexpr int kResColsPerBlock = kThreads * 8;  // 1024
constexpr int kResMaxCluster = 8;

__global__ void __launch_bounds__(kThreads, 8) combine_residual_kernel(
    const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_row, const float* __restrict__ topk_w,
    const uint16_t* __restrict__ gain, float eps, float keep, float add, uint16_t* __restrict__ resid, int T, int d,
    int K, int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float warp_ss[kThreads / 32];
  __shared__ float block_ss;
  __shared__ float inv_r;
  const int nb = static_cast<int>(cluster.num_blocks());  // column blocks of the row
  const int t = static_cast<int>(blockIdx.x) / nb;
  const int cb = static_cast<int>(cluster.block_rank());
  const int c = cb * kResColsPerBlock + threadIdx.x * 8;
  const bool active = c < d;  // no early return: every thread meets the cluster barrier
  const int64_t R = static_cast<int64_t>(T) * K;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < K; k0 += kMaxK) {
    const int nk = min(kMaxK, K - k0);
    uint4 v[kMaxK];
    float w[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      w[k] = 0.f;
      if (k < nk) {
        const int r = inv_row[static_cast<size_t>(t) * K + k0 + k];
        if (r < 0 || r >= R) {
          if (threadIdx.x == 0 && cb == 0) latch_status(status, MOE_DEV_BAD_ROW);
        } else if (active) {
          w[k] = topk_w[static_cast<size_t>(t) * K + k0 + k];
          v[k] = *reinterpret_cast<const uint4*>(y + static_cast<size_t>(r) * d + c);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {  // slot order
      if (k < nk) {
        fma_bf16x2(v[k].x, w[k], acc[0], acc[1]);
        fma_bf16x2(v[k].y, w[k], acc[2], acc[3]);
        fma_bf16x2(v[k].z, w[k], acc[4], acc[5]);
        fma_bf16x2(v[k].w, w[k], acc[6], acc[7]);
      }
    }
  }
  uint4 h = make_uint4(0, 0, 0, 0), g = make_uint4(0, 0, 0, 0);
  if (active) {  // in flight across the reduction
    h = *reinterpret_cast<const uint4*>(resid + static_cast<size_t>(t) * d + c);
    g = *reinterpret_cast<const uint4*>(gain + c);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(acc[i], acc[i], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int i = 0; i < kThreads / 32; ++i) b += warp_ss[i];
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
    const uint32_t hv[4] = {h.x, h.y, h.z, h.w}, gv[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float n0 = acc[2 * i] * ir * __uint_as_float(gv[i] << 16);
      const float n1 = acc[2 * i + 1] * ir * __uint_as_float(gv[i] & 0xFFFF0000u);
      const float h0 = fmaf(keep, __uint_as_float(hv[i] << 16), add * n0);
      const float h1 = fmaf(keep, __uint_as_float(hv[i] & 0xFFFF0000u), add * n1);
      const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
      o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(resid + static_cast<size_t>(t) * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // no block leaves while another may still read it
}

}  // namespace

cudaError_t launch_combine_residual(const uint16_t* y_perm, const int32_t* inv_row, const float* topk_w,
                                    const uint16_t* gain, float eps, int step, uint16_t* resid, int T, int d,
                                    int top_k, int32_t* status, cudaStream_t stream) {
  const int nb = (d + kResColsPerBlock - 1) / kResColsPerBlock;
  if (nb > kResMaxCluster) return cudaErrorInvalidValue;  // d > 8192
  const float keep = static_cast<float>(sqrt(static_cast<double>(step - 1) / step));
  const float add = static_cast<float>(1.0 / sqrt(static_cast<double>(step)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(T) * nb));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nb;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_residual_kernel, y_perm, inv_row, topk_w, gain, eps, keep, add, resid, T, d,
                            top_k, status);
}

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_row, const float* topk_w, uint16_t* out,
                           int T, int d, int top_k, int32_t* status, cudaStream_t stream) {
  dim3 grid(T, (d / 8 + kThreads - 1) / kThreads);
  combine_kernel<<<grid, kThreads, 0, stream>>>(y_perm, inv_row, topk_w, out, T, d, top_k, status);
  return cudaGetLastError();
}

}  // namespace beammoe
