// Work schedule of the expert GEMMs, built on the device from the expert
// offsets (by the expert FFN's schedule kernel or the small-batch plan kernel
// of the permutation) and read by every role of the GEMM kernels.
//
// The schedule is one int4 per expert and the expert of every token tile, not
// a list of work items: an item follows from two loads, so building the
// schedule writes E entries (4 KB at E = 256) and one int per token tile
// instead of one 16-byte item per (expert, weight tile, token tile).
#pragma once

#include "common.cuh"

namespace beammoe {

struct ScheduleArgs {
  int n_max;        // tokens per tile at most (multiple of 16)
  int wt1, wt2;     // weight tiles per expert in GEMM1 and GEMM2
  int R;            // rows (T * top_k)
  int4* table;      // [E] {token tiles before expert e, first row, rows, rows per tile}
  int32_t* tile_expert;  // [max_tiles] expert of each token tile
  int max_tiles;
  int32_t* n_items; // [2] work items of GEMM1 and GEMM2
};

// Called by every thread of the block (blockDim.x a multiple of 32, >= E):
// thread e takes expert e. Tokens of an expert are split into ceil(n/n_max)
// tiles of near-equal size (multiples of 16). `offsets` may be in shared or
// global memory; `warp_sums` is shared scratch of blockDim.x / 32 ints.
// Offsets that are not a non-decreasing split of [0, R] latch MOE_DEV_BAD_ROW
// and give the expert no work.
__device__ inline void build_schedule(const int32_t* offsets, int E, const ScheduleArgs& s, int32_t* status,
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
  const int tile0 = base + incl - ntiles;  // token tiles before this expert
  if (e < E) s.table[e] = make_int4(tile0, row0, n, tsz);
  if (!dcheck(total <= s.max_tiles, status)) ntiles = 0;
  for (int j = 0; j < ntiles; ++j) s.tile_expert[tile0 + j] = e;
  if (threadIdx.x == 0) {
    s.n_items[0] = total * s.wt1;
    s.n_items[1] = total * s.wt2;
  }
}

// Work item `it` (< the GEMM's item count) of a GEMM whose experts have `wt`
// weight tiles each: {expert, weight tile, first row, tokens}. Items run expert
// by expert, inside an expert weight tile by weight tile, inside a weight tile
// token tile by token tile, so the token tiles of one weight tile run side by
// side and share it through L2. Expert e owns items [tile0, tile0 + tiles) x wt,
// so item `it` lies in the expert of token tile it / wt.
__device__ __forceinline__ int4 work_item(const int4* __restrict__ table, const int32_t* __restrict__ tile_expert,
                                          int wt, int it) {
  const int e = __ldg(tile_expert + it / wt);
  const int4 t = __ldg(table + e);
  const int ntiles = max((t.z + t.w - 1) / t.w, 1);
  const int local = it - t.x * wt;
  const int w = local / ntiles, j = local - w * ntiles;
  return make_int4(e, w, t.y + j * t.w, min(t.w, t.z - j * t.w));
}

}  // namespace beammoe
