// Permutation of the Beam MoE block: the (token, slot) pairs routed to each
// expert are grouped into consecutive rows, tokens ascending inside an
// expert, and the activations are gathered into that order for the expert
// GEMMs.
//
// Method (no sort): a token x expert bitmap is built from the routing
// (one bit per token per expert). A token's row inside expert e is the number
// of set bits before it in e's bitmap column, so the per-word popcount prefix
// sums of each column give every row directly and deterministically.
//   1. bitmap_kernel     set bit (e, t) for every slot            T*K threads
//   2. column_scan_kernel per expert: popcount prefix over words   E blocks
//   3. offsets_kernel    exclusive scan of the counts              1 block
//   4. gather_kernel     rows, inverse rows, x -> x_perm copy      1 block/token, 1 warp/slot
#include "common.cuh"
#include "kernels.h"

namespace beammoe {

namespace {

__global__ void bitmap_kernel(const int32_t* __restrict__ idx, int T, int E, int K, int nw,
                              uint32_t* __restrict__ bitmap, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * K) return;
  const int t = static_cast<int>(i / K);
  const int e = idx[i];
  if (e < 0 || e >= E) {
    latch_status(status, MOE_DEV_BAD_EXPERT);
    return;
  }
  const uint32_t bit = 1u << (t & 31);
  // a bit already set means another slot of this token named the same expert
  if (atomicOr(bitmap + static_cast<size_t>(e) * nw + (t >> 5), bit) & bit)
    latch_status(status, MOE_DEV_DUP_EXPERT);
}

// One block per expert: word_prefix[e][w] = set bits of column e before word w.
__global__ void __launch_bounds__(256) column_scan_kernel(const uint32_t* __restrict__ bitmap, int nw,
                                                          int32_t* __restrict__ word_prefix,
                                                          int32_t* __restrict__ counts) {
  __shared__ int32_t warp_sums[8];
  pdl_launch_dependents();
  pdl_wait();
  const int e = blockIdx.x;
  const uint32_t* col = bitmap + static_cast<size_t>(e) * nw;
  int32_t* pre = word_prefix + static_cast<size_t>(e) * nw;
  const int per = (nw + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * per;
  int local = 0;
  for (int w = w0; w < w0 + per && w < nw; ++w) local += __popc(col[w]);
  // block exclusive scan of `local`
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int warp_base = 0;
  for (int i = 0; i < warp; ++i) warp_base += warp_sums[i];
  int run = warp_base + incl - local;
  for (int w = w0; w < w0 + per && w < nw; ++w) {
    pre[w] = run;
    run += __popc(col[w]);
  }
  if (threadIdx.x == blockDim.x - 1) {
    int total = 0;
    for (int i = 0; i < 8; ++i) total += warp_sums[i];
    counts[e] = total;
  }
}

// offsets[e] = sum of counts[0..e), offsets[E] = total (single block, E <= 1024).
__global__ void __launch_bounds__(1024) offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                       int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_sums[32];
  pdl_launch_dependents();
  pdl_wait();
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const int v = (i < E) ? counts[i] : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_sums[w];
  if (i < E) offsets[i] = base + incl - v;
  if (i == E - 1) offsets[E] = base + incl;
}

// One block per token, one warp per slot (slots k, k + 8, ...): the slot's row,
// then x[t] copied to it. A block per token keeps small batches spread over
// the whole GPU.
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(32 * kGatherWarps) gather_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ idx, int T, int d, int E, int K, int nw,
    const uint32_t* __restrict__ bitmap, const int32_t* __restrict__ word_prefix,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ row_token, int32_t* __restrict__ inv_row,
    uint16_t* __restrict__ x_perm) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  const int nvec = d / 8;
  for (int k = warp; k < K; k += kGatherWarps) {
    int my_row = -1;
    if (lane == 0) {
      const int e = idx[static_cast<size_t>(t) * K + k];
      if (e >= 0 && e < E) {
        const size_t wi = static_cast<size_t>(e) * nw + (t >> 5);
        const uint32_t below = bitmap[wi] & ((1u << (t & 31)) - 1u);
        my_row = offsets[e] + word_prefix[wi] + __popc(below);
        row_token[my_row] = t;
      }
      inv_row[static_cast<size_t>(t) * K + k] = my_row;
    }
    const int r = __shfl_sync(0xffffffffu, my_row, 0);  // whole warp, outside the lane-strided loop
    if (r < 0) continue;
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(r) * d);
    for (int c = lane; c < nvec; c += 32) dst[c] = src[c];
  }
}

}  // namespace

int bitmap_words(int T) { return (T + 31) / 32; }

size_t bitmap_bytes(int T, int E) { return sizeof(uint32_t) * static_cast<size_t>(E) * bitmap_words(T); }

cudaError_t launch_permute(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int top_k,
                           uint32_t* bitmap, int32_t* word_prefix, int32_t* counts, int32_t* offsets,
                           int32_t* row_token, int32_t* inv_row, uint16_t* x_perm, int32_t* status,
                           cudaStream_t stream, bool bitmap_zeroed) {
  const int nw = bitmap_words(T);
  cudaError_t err = cudaSuccess;
  if (!bitmap_zeroed && (err = cudaMemsetAsync(bitmap, 0, bitmap_bytes(T, E), stream)) != cudaSuccess) return err;
  const int64_t slots = static_cast<int64_t>(T) * top_k;
  if ((err = launch_pdl(bitmap_kernel, dim3(static_cast<unsigned>((slots + 255) / 256)), dim3(256), 0, stream, topk_idx,
                        T, E, top_k, nw, bitmap, status)) != cudaSuccess)
    return err;
  if ((err = launch_pdl(column_scan_kernel, dim3(E), dim3(256), 0, stream, bitmap, nw, word_prefix, counts)) !=
      cudaSuccess)
    return err;
  if ((err = launch_pdl(offsets_kernel, dim3(1), dim3(1024), 0, stream, counts, E, offsets)) != cudaSuccess) return err;
  return launch_pdl(gather_kernel, dim3(T), dim3(32 * kGatherWarps), 0, stream, x, topk_idx, T, d, E, top_k, nw,
                    bitmap, word_prefix, offsets, row_token, inv_row, x_perm);
}

}  // namespace beammoe
