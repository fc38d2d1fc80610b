// Combine of the Beam MoE block (release article, section "Mixture of
// Experts": expert outputs summed with the normalised router weights, scaled
// by 2.5 -- the scale is already inside topk_w -- and no shared expert).
//
// out[t][c] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*K+k]][c] ), the sum
// in FP32 in slot order (deterministic, no atomics). Each thread owns eight
// consecutive columns: one 16-byte load of every slot's bf16 row (all K loads
// issued before the first use), two 8-byte stores. HBM-bound: K*d*2 bytes
// read and d*2 written per token.
#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 16;

__device__ __forceinline__ void fma_bf16x2(uint32_t v, float w, float& a, float& b) {
  a = fmaf(w, __uint_as_float(v << 16), a);
  b = fmaf(w, __uint_as_float(v & 0xFFFF0000u), b);
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ y,
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

}  // namespace

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_row, const float* topk_w, uint16_t* out,
                           int T, int d, int top_k, int32_t* status, cudaStream_t stream) {
  dim3 grid(T, (d / 8 + kThreads - 1) / kThreads);
  combine_kernel<<<grid, kThreads, 0, stream>>>(y_perm, inv_row, topk_w, out, T, d, top_k, status);
  return cudaGetLastError();
}

}  // namespace beammoe
