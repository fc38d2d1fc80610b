// Work items of the expert GEMMs, built on the device from the expert offsets
// (shared by the expert FFN's schedule kernel and the small-batch plan kernel
// of the permutation).
#pragma once

#include "common.cuh"

namespace beammoe {

// Where the work items go and how tokens are cut into tiles.
struct ScheduleArgs {
  int n_max;        // tokens per tile at most (multiple of 16)
  int wt1, wt2;     // weight tiles per expert in GEMM1 and GEMM2
  int R;            // rows (T * top_k)
  int4* items1;     // GEMM1 work items {expert, weight tile, first row, tokens}
  int4* items2;     // GEMM2 work items
  int32_t* n_items; // [2]
  int64_t cap1, cap2;  // item capacity of items1 / items2 (checked by the debug build)
};

// Called by every thread of the block (blockDim.x a multiple of 32, >= E):
// thread e takes expert e. Tokens of an expert are split into ceil(n/n_max)
// tiles of near-equal size (multiples of 16). Items are ordered expert, weight
// tile, token tile so the token tiles of one weight tile run side by side and
// share it through L2. `offsets` may be in shared or global memory;
// `warp_sums` is shared scratch of blockDim.x / 32 ints. Offsets that are not
// a non-decreasing split of [0, R] latch MOE_DEV_BAD_ROW and give the expert
// no work.
__device__ inline void build_work_items(const int32_t* offsets, int E, const ScheduleArgs& s, int32_t* status,
                                        int* warp_sums) {
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5, nwarps = blockDim.x >> 5;
  int n = 0, row0 = 0, ntiles = 0, tsz = 16;
  if (e < E) {
    const int a = offsets[e], b = offsets[e + 1];
    if (a < 0 || b < a || b > s.R) {
      latch_status(status, MOE_DEV_BAD_ROW);
    } else {
      n = b - a;
      row0 = a;
    }
    if (n > 0) {
      ntiles = (n + s.n_max - 1) / s.n_max;
      tsz = ((n + ntiles - 1) / ntiles + 15) & ~15;
      if (tsz > s.n_max) tsz = s.n_max;
      ntiles = (n + tsz - 1) / tsz;
    }
  }
  int incl = ntiles;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();  // warp_sums may still be read from an earlier use
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < nwarps; ++w) {
    if (w < warp) base += warp_sums[w];
    total += warp_sums[w];
  }
  const int tile0 = base + incl - ntiles;  // tiles before this expert
  if (!dcheck(static_cast<int64_t>(total) * s.wt1 <= s.cap1 && static_cast<int64_t>(total) * s.wt2 <= s.cap2, status))
    ntiles = 0;
  for (int wt = 0; wt < s.wt1; ++wt)
    for (int j = 0; j < ntiles; ++j)
      s.items1[static_cast<size_t>(tile0) * s.wt1 + wt * ntiles + j] =
          make_int4(e, wt, row0 + j * tsz, min(tsz, n - j * tsz));
  for (int wt = 0; wt < s.wt2; ++wt)
    for (int j = 0; j < ntiles; ++j)
      s.items2[static_cast<size_t>(tile0) * s.wt2 + wt * ntiles + j] =
          make_int4(e, wt, row0 + j * tsz, min(tsz, n - j * tsz));
  if (threadIdx.x == 0) {
    s.n_items[0] = total * s.wt1;
    s.n_items[1] = total * s.wt2;
  }
}

}  // namespace beammoe
