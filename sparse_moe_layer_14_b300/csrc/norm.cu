// Pre-norm of the MoE sublayer input (release article, section "Residual
// stream": every sublayer is normalised before and after, with the norms in
// FP32):
//
//   x[t][c] = bf16( h[t][c] * inv_r * gain[c] ),  inv_r = 1 / sqrt(mean_c(h[t][c]^2) + eps)
//
// One block per token row. Each thread sums the squares of its 16-byte
// vectors in FP32; the warps reduce with shuffles and every thread adds the
// warp partials in the same order. The scaled pass re-reads the row (10 KB at
// d = 5120, an L1/L2 hit), so HBM sees 2d bytes read and 2d written per token.
#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

constexpr int kNormThreads = 128;

__device__ __forceinline__ float lo_bf16(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// bf16x2 word of (h * inv_r * g) for the two elements of the words v and g
__device__ __forceinline__ uint32_t scale_pair(uint32_t v, uint32_t g, float inv_r) {
  const __nv_bfloat162 b =
      __floats2bfloat162_rn(lo_bf16(v) * inv_r * lo_bf16(g), hi_bf16(v) * inv_r * hi_bf16(g));
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(kNormThreads) pre_norm_kernel(const uint16_t* __restrict__ h,
                                                                const uint16_t* __restrict__ gain, float eps,
                                                                int d, uint16_t* __restrict__ x) {
  pdl_launch_dependents();
  pdl_wait();
  const int nv = d >> 3;  // 16-byte vectors per row (d is a multiple of 64)
  const uint4* row = reinterpret_cast<const uint4*>(h + static_cast<size_t>(blockIdx.x) * d);
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += kNormThreads) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = lo_bf16(w[j]), b = hi_bf16(w[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float part[kNormThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) total += part[i];
  const float inv_r = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
  const uint4* g4 = reinterpret_cast<const uint4*>(gain);
  uint4* out = reinterpret_cast<uint4*>(x + static_cast<size_t>(blockIdx.x) * d);
  for (int i = threadIdx.x; i < nv; i += kNormThreads) {
    const uint4 v = row[i], g = __ldg(g4 + i);
    out[i] = make_uint4(scale_pair(v.x, g.x, inv_r), scale_pair(v.y, g.y, inv_r), scale_pair(v.z, g.z, inv_r),
                        scale_pair(v.w, g.w, inv_r));
  }
}

}  // namespace

cudaError_t launch_pre_norm(const uint16_t* h, const uint16_t* gain, float eps, uint16_t* x, int T, int d,
                            cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  return launch_pdl(pre_norm_kernel, dim3(T), dim3(kNormThreads), 0, stream, h, gain, eps, d, x);
}

}  // namespace beammoe
