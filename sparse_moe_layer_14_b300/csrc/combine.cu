// Combine of the Beam MoE block (release article, section "Mixture of
// Experts": expert outputs summed with the normalised router weights, scaled
// by 2.5 -- the scale is already inside topk_w -- and no shared expert).
//
// out[t][c] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*K+k]][c] ), the sum
// in FP32 in slot order (deterministic, no atomics). Each thread owns four
// consecutive columns: 16-byte loads of every slot's row, an 8-byte store.
#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) combine_kernel(const float* __restrict__ y,
                                                           const int32_t* __restrict__ inv_row,
                                                           const float* __restrict__ topk_w,
                                                           uint16_t* __restrict__ out, int T, int d, int K,
                                                           int32_t* status) {
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kThreads + threadIdx.x) * 4;
  if (c >= d) return;
  const int64_t R = static_cast<int64_t>(T) * K;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < K; ++k) {
    const int r = inv_row[static_cast<size_t>(t) * K + k];
    if (r < 0 || r >= R) {
      if (c == 0) latch_status(status, MOE_DEV_BAD_ROW);
      continue;
    }
    const float w = topk_w[static_cast<size_t>(t) * K + k];
    const float4 v = *reinterpret_cast<const float4*>(y + static_cast<size_t>(r) * d + c);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d + c) = pk;
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* inv_row, const float* topk_w, uint16_t* out,
                           int T, int d, int top_k, int32_t* status, cudaStream_t stream) {
  dim3 grid(T, (d / 4 + kThreads - 1) / kThreads);
  combine_kernel<<<grid, kThreads, 0, stream>>>(y_perm, inv_row, topk_w, out, T, d, top_k, status);
  return cudaGetLastError();
}

}  // namespace beammoe
