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
//   4. gather_kernel     rows, inverse rows, x -> x_perm copy      1 block per (token, slot)
// Small batches (E * ceil(T/32) words fit in shared memory) do 1-3 in one CTA,
// plan_small_kernel, which needs no cleared bitmap in global memory and can
// also build the expert GEMMs' work schedule.
#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"

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

// offsets[e] = sum of counts[0..e), offsets[E] = total (single block, E <= 1024);
// with `do_schedule` also the expert GEMMs' work schedule from them.
__global__ void __launch_bounds__(1024) offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                       int32_t* __restrict__ offsets, ScheduleArgs sched,
                                                       int do_schedule, int32_t* status) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t offs[257];
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
  if (!do_schedule) return;
  if (i < E) offs[i] = base + incl - v;  // do_schedule implies E <= 256
  if (i == E - 1) offs[E] = base + incl;
  __syncthreads();  // every offset is in shared memory before any thread reads its neighbour's
  build_schedule(offs, E, sched, status, warp_sums);
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxWords = 8192;  // 32 KB of bitmap: T <= 1024 at E = 256

// One CTA: the bitmap in shared memory (set bits, repeats latched), then one
// warp per expert column for the per-word prefix counts (written with the
// bitmap words for the gather) and the count, an exclusive scan of the counts
// for the offsets, and with `do_schedule` the work schedule of the expert GEMMs.
__global__ void __launch_bounds__(kPlanThreads) plan_small_kernel(
    const int32_t* __restrict__ idx, int T, int E, int K, int nw, uint32_t* __restrict__ bitmap,
    int32_t* __restrict__ word_prefix, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* status, ScheduleArgs sched, int do_schedule) {
  __shared__ uint32_t bm[kPlanMaxWords];
  __shared__ int32_t cnt[256];
  __shared__ int32_t offs[257];
  __shared__ int warp_sums[32];
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int nwords = E * nw;
  for (int i = threadIdx.x; i < nwords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int slots = T * K;
  for (int i = threadIdx.x; i < slots; i += blockDim.x) {
    const int t = i / K, e = idx[i];
    if (e < 0 || e >= E) {
      latch_status(status, MOE_DEV_BAD_EXPERT);
      continue;
    }
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bm[e * nw + (t >> 5)], bit) & bit) latch_status(status, MOE_DEV_DUP_EXPERT);
  }
  __syncthreads();
  for (int e = warp; e < E; e += nwarps) {
    int run = 0;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t v = w < nw ? bm[e * nw + w] : 0u;
      const int c = __popc(v);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (w < nw) {
        word_prefix[static_cast<size_t>(e) * nw + w] = run + incl - c;
        bitmap[static_cast<size_t>(e) * nw + w] = v;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cnt[e] = run;
  }
  __syncthreads();
  {  // offsets: exclusive scan of the counts
    const int i = threadIdx.x;
    const int v = i < E ? cnt[i] : 0;
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
    if (i < E) {
      offs[i] = base + incl - v;
      counts[i] = v;
      offsets[i] = base + incl - v;
    }
    if (i == E - 1) {
      offs[E] = base + incl;
      offsets[E] = base + incl;
    }
    __syncthreads();
  }
  if (do_schedule) build_schedule(offs, E, sched, status, warp_sums);
}

// One block per (token, slot): every thread derives the slot's row from the
// bitmap (the same few loads, served to the whole block at once), thread 0
// records it in row_token and inv_row, and the block copies x[t] to it with
// 16-byte loads, all issued before the stores.
constexpr int kGatherThreads = 128;

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ idx, int T, int d, int E, int K, int nw,
    const uint32_t* __restrict__ bitmap, const int32_t* __restrict__ word_prefix,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ row_token, int32_t* __restrict__ inv_row,
    uint16_t* __restrict__ x_perm, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t slot = blockIdx.x;
  const int t = static_cast<int>(slot / K);
  const int e = idx[slot];
  int row = -1;
  if (e >= 0 && e < E) {
    const size_t wi = static_cast<size_t>(e) * nw + (t >> 5);
    const uint32_t below = bitmap[wi] & ((1u << (t & 31)) - 1u);
    row = offsets[e] + word_prefix[wi] + __popc(below);
    if (!dcheck(row >= 0 && row < T * K, status)) row = -1;
  }
  if (threadIdx.x == 0) {
    if (row >= 0) row_token[row] = t;
    inv_row[slot] = row;
  }
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(row) * d);
  const int nvec = d / 8;
  constexpr int kUnroll = 4;
  for (int c0 = threadIdx.x; c0 < nvec; c0 += kUnroll * kGatherThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * kGatherThreads;
      if (c < nvec) v[u] = src[c];
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * kGatherThreads;
      if (c < nvec) dst[c] = v[u];
    }
  }
}

}  // namespace

int bitmap_words(int T) { return (T + 31) / 32; }

size_t bitmap_bytes(int T, int E) { return sizeof(uint32_t) * static_cast<size_t>(E) * bitmap_words(T); }

bool permute_uses_plan_kernel(int T, int E) {
  return E <= 256 && static_cast<int64_t>(E) * bitmap_words(T) <= kPlanMaxWords;
}

cudaError_t launch_permute(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int top_k,
                           uint32_t* bitmap, int32_t* word_prefix, int32_t* counts, int32_t* offsets,
                           int32_t* row_token, int32_t* inv_row, uint16_t* x_perm, int32_t* status,
                           cudaStream_t stream, bool bitmap_zeroed, const ScheduleArgs* sched) {
  const int nw = bitmap_words(T);
  cudaError_t err = cudaSuccess;
  if (permute_uses_plan_kernel(T, E)) {
    ScheduleArgs none{};
    if ((err = launch_pdl(plan_small_kernel, dim3(1), dim3(kPlanThreads), 0, stream, topk_idx, T, E, top_k, nw,
                          bitmap, word_prefix, counts, offsets, status, sched ? *sched : none,
                          sched ? 1 : 0)) != cudaSuccess)
      return err;
    return launch_pdl(gather_kernel, dim3(static_cast<unsigned>(static_cast<int64_t>(T) * top_k)),
                      dim3(kGatherThreads), 0, stream, x, topk_idx, T, d, E, top_k, nw, bitmap, word_prefix, offsets,
                      row_token, inv_row, x_perm, status);
  }
  if (!bitmap_zeroed && (err = cudaMemsetAsync(bitmap, 0, bitmap_bytes(T, E), stream)) != cudaSuccess) return err;
  const int64_t slots = static_cast<int64_t>(T) * top_k;
  if ((err = launch_pdl(bitmap_kernel, dim3(static_cast<unsigned>((slots + 255) / 256)), dim3(256), 0, stream, topk_idx,
                        T, E, top_k, nw, bitmap, status)) != cudaSuccess)
    return err;
  if ((err = launch_pdl(column_scan_kernel, dim3(E), dim3(256), 0, stream, bitmap, nw, word_prefix, counts)) !=
      cudaSuccess)
    return err;
  ScheduleArgs none{};
  if ((err = launch_pdl(offsets_kernel, dim3(1), dim3(1024), 0, stream, counts, E, offsets, sched ? *sched : none,
                        sched && E <= 256 ? 1 : 0, status)) != cudaSuccess)
    return err;
  return launch_pdl(gather_kernel, dim3(static_cast<unsigned>(static_cast<int64_t>(T) * top_k)),
                    dim3(kGatherThreads), 0, stream, x, topk_idx, T, d, E, top_k, nw, bitmap, word_prefix, offsets,
                    row_token, inv_row, x_perm, status);
}

}  // namespace beammoe
