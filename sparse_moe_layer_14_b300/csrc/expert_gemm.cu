// Expert SwiGLU MLPs of the Beam MoE block as two grouped GEMMs on the
// sm_103a tensor cores (release article, section "Mixture of Experts": each
// expert is a SwiGLU MLP with intermediate size 2,560; the NVFP4 checkpoint
// stores most parameters in 4-bit precision for Blackwell; section "Residual
// stream": the SwiGLU product is computed in FP32).
//
//   GEMM1 + SwiGLU:  h[r][i] = bf16( silu(x_perm[r].Wg_e[i]) * (x_perm[r].Wu_e[i]) )
//   GEMM2:           y[r][n] = h[r] . Wd_e[n]   (FP32; bf16 for the dense MLP's output)
//
// Every work item runs two 128-row weight tiles against the same token tile
// (two MMAs per K step sharing the token operand): the gate and up tiles of
// the same 128 intermediate rows in GEMM1, two consecutive 128-row tiles of
// W_down (256 output columns) in GEMM2.
//
// Design (weight-stationary, "swap AB"): the MMA's M operand is a 128-row
// tile of one expert's weights (K-major, straight from the checkpoint
// layout) and its N operand is the expert's tokens (rows of x_perm / h),
// N = the tile's token count rounded up to 16, so a decode batch with two or
// three tokens per expert does no padded tensor work and every weight byte is
// streamed from HBM once per token tile. Accumulators live in TMEM:
// D[weight row][token], fp32.
//
// One persistent CTA per SM:
//   warp 0      TMA producer: weight tile(s) + token rows per 64-wide K slice
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2..9  epilogue, two warpgroups splitting the token columns:
//               tcgen05.ld, SwiGLU in FP32 (GEMM1) or the FP32 expert output
//               (GEMM2; bf16 for the dense MLP)
//   warps 10..17 (NVFP4 and FP8 weights) converters: e2m1 codes times their
//               e4m3 block scale (exact in bf16), or e4m3 codes times their
//               fp32 block scale (rounded once to bf16), written to tensor
//               memory, from where the MMA reads its A operand; the NVFP4 fp32
//               tensor scale is applied to the accumulator in the epilogue.
//               The TMA ring holds packed codes and token rows; decoded tiles
//               cycle through 2-4 TMEM slots. (Decoded tiles staged in shared
//               memory instead, read like bf16 tiles, measured slower.)
// Waits off the critical path sleep between polls: the MMA issuer shares a
// scheduler with epilogue and converter warps, and their spinning took its
// issue slots (MMA slices up to 1.5x slower).
// Work items {expert, weight tile, first row, tokens} follow from a per-expert
// schedule built on the device from the expert offsets (no host
// synchronisation) and are taken round-robin.
// Every mbarrier wait is bounded; on expiry the CTA latches MOE_DEV_TIMEOUT,
// waits (bounded) for its own copies and MMAs in flight, frees TMEM, returns.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"

namespace beammoe {

namespace {

constexpr int BM = 128;       // weight rows per tile = MMA M
constexpr int BK = 64;        // K elements per pipeline stage (128 bytes of bf16)
constexpr int TOK_BOX = 16;   // token rows per TMA box
constexpr int kMaxStages = 8;
constexpr int kMaxAcc = 4;
constexpr int kMaxConv = 4;   // decoded-weight slots in TMEM
// TMEM columns of one slot: a K slice (64 elements) of both weight tiles, tile 0 in columns
// [0, 32), tile 1 in [32, 64) (two bf16 a column)
constexpr int kConvCols = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kATileBytes = BM * BK * 2;            // 16 KB bf16 weight tile
constexpr uint32_t kPTileBytes = BM * BK / 2;            // 4 KB packed e2m1 weight tile
constexpr uint32_t kP8TileBytes = BM * BK;               // 8 KB e4m3 weight tile
// Weight formats of the kernel (moe_wfmt_t values): bf16 straight from TMA into the
// MMA; NVFP4 and FP8 through the converter warps into tensor memory.
constexpr int kFmtBf16 = 0, kFmtNvfp4 = 1, kFmtFp8 = 2;
constexpr uint32_t kTokBoxBytes = TOK_BOX * BK * 2;      // 2 KB
constexpr uint64_t kDrainNs = 1000000000ull;             // 1 s bound for draining on abort
constexpr uint64_t kWaitNs = 2000000000ull;              // 2 s bound of a pipeline wait
constexpr int kSmemLimit = 232448;                       // 227 KB opt-in per block
// Sleep between polls of a wait off the critical path (nanoseconds): the producer and
// converters wait a slot at a time, the epilogue a whole item. The single thread that issues
// the MMAs never sleeps; it shares a scheduler with two epilogue warps (and with converter
// warps), and spinning neighbours would take its issue slots.
constexpr unsigned kSleepSlotNs = 32, kSleepItemNs = 512;

constexpr int kEpiThreads = 256;    // two epilogue warpgroups
constexpr int kConvBase = 320;      // first converter thread (NVFP4)
constexpr int kConvThreads = 256;   // one converter thread per row of each weight tile (NVFP4)
constexpr int threads_for(int fmt) { return fmt != kFmtBf16 ? kConvBase + kConvThreads : 320; }

struct GemmArgs {
  const int4* table;       // work schedule (schedule.cuh)
  const int32_t* tile_expert;
  int wt;                  // weight tiles per expert
  const int32_t* n_items;
  int K;           // reduction length
  int Nw;          // weight rows per expert = output columns
  int E;           // experts
  int R;           // rows of the token operand (T * top_k)
  int n_max;       // max tokens per item (multiple of 16)
  int stages;
  int acc_bufs;
  int acc_cols;    // TMEM columns per accumulator buffer
  uint32_t stage_bytes;
  uint32_t b_offset;  // token tile offset inside a stage
  uint32_t p_offset;  // packed weight tile offset inside a stage (NVFP4)
  uint32_t a_col;     // first TMEM column of the decoded weight slots (NVFP4, FP8)
  int conv_stages;
  uint16_t* h_out;    // GEMM1 output [R][Nw] bf16
  uint16_t* y_out;    // GEMM2 output [R][Nw] bf16 (the dense MLP's output), or null
  float* y_f32;       // GEMM2 output [R][Nw] fp32 (the experts' outputs), or null
  const float* ts0;   // per-expert scale applied to accumulator 0 (NVFP4), or null
  const float* ts1;
  const uint8_t* sf0;  // e4m3 block scales [E*Nw][K/16] of matrix 0 (NVFP4)
  const uint8_t* sf1;
  const float* fs0;    // fp32 block scales [E][Nw/128][K/128] of matrix 0 (FP8)
  const float* fs1;
  int32_t* status;
  int32_t* timeout_where;
  long long wait_spins;
};

__device__ __forceinline__ void fail(const GemmArgs& p, volatile int* abort, int where) {
  latch_status(p.status, MOE_DEV_TIMEOUT);
  if (p.timeout_where) atomicCAS(p.timeout_where, 0, where);
  *abort = 1;
}

// 8 e2m1 codes (one 32-bit word, element 2j in the low nibble of byte j) times
// one e4m3 scale (broadcast in both halves of `scale2`, as f16x2) -> 8 bf16,
// returned as four bf16x2 words in element order. Every product has at most
// 6 significant bits, so f16 and bf16 represent it exactly.
__device__ __forceinline__ uint4 decode8(uint32_t codes, uint32_t scale2) {
  uint32_t h[4];
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t prod;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(prod) : "r"(h[i]), "r"(scale2));
    const __half2 ph = *reinterpret_cast<const __half2*>(&prod);
    const __nv_bfloat162 b = __floats2bfloat162_rn(__low2float(ph), __high2float(ph));
    out[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// e4m3 scale byte -> (s, s) as f16x2.
__device__ __forceinline__ uint32_t scale_pair(uint32_t byte) {
  const uint16_t two = static_cast<uint16_t>(byte * 0x0101u);
  uint32_t s;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s) : "h"(two));
  return s;
}

// Decode half h of row r of one packed 128 x 64 weight tile (the row's 64
// e2m1 codes are 32 bytes; half h is elements 32h..32h+31, bytes 16h..16h+15)
// with its two e4m3 block scales (bytes 2h and 2h+1 of `sc`, the row's four
// scales of the slice) into 16 bf16x2 words in element order: word c holds
// elements 32h + 2c (low half) and 32h + 2c + 1.
__device__ __forceinline__ void decode_half(const uint8_t* packed_tile, int r, int h, uint32_t sc,
                                            uint32_t (&out)[16]) {
  const uint4 p = *reinterpret_cast<const uint4*>(packed_tile + r * 32 + h * 16);
  const uint32_t s2a = scale_pair((sc >> (16 * h)) & 0xFFu), s2b = scale_pair((sc >> (16 * h + 8)) & 0xFFu);
  const uint4 v0 = decode8(p.x, s2a), v1 = decode8(p.y, s2a), v2 = decode8(p.z, s2b), v3 = decode8(p.w, s2b);
  out[0] = v0.x, out[1] = v0.y, out[2] = v0.z, out[3] = v0.w;
  out[4] = v1.x, out[5] = v1.y, out[6] = v1.z, out[7] = v1.w;
  out[8] = v2.x, out[9] = v2.y, out[10] = v2.z, out[11] = v2.w;
  out[12] = v3.x, out[13] = v3.y, out[14] = v3.z, out[15] = v3.w;
}

// Two e4m3 codes (low byte = lower element) times the fp32 block scale `s`:
// e4m3 -> f16 is exact, the product is rounded to fp32 and then to bf16.
__device__ __forceinline__ uint32_t e4m3x2_scaled_bf16x2(uint32_t two, float s) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two)));
  const __half2 ph = *reinterpret_cast<const __half2*>(&h);
  const __nv_bfloat162 b = __floats2bfloat162_rn(__low2float(ph) * s, __high2float(ph) * s);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Half h of row r of one 128 x 64 FP8 weight tile (64 e4m3 codes, element k in
// byte k; half h is bytes 32h..32h+31) scaled and rounded as above: 16 bf16x2
// words in element order.
__device__ __forceinline__ void decode_half_fp8(const uint8_t* packed_tile, int r, int h, float s,
                                                uint32_t (&out)[16]) {
  const uint4* row = reinterpret_cast<const uint4*>(packed_tile + r * 64 + h * 32);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 p = row[q];
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[8 * q + 2 * i] = e4m3x2_scaled_bf16x2(w[i] & 0xFFFFu, s);
      out[8 * q + 2 * i + 1] = e4m3x2_scaled_bf16x2(w[i] >> 16, s);
    }
  }
}

template <bool kGLU, int kFmt>
__global__ void __launch_bounds__(threads_for(kFmt), 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB64,
                       const __grid_constant__ CUtensorMap tmB128, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t conv_bar[kMaxStages];        // decoded slot ready (NVFP4)
  __shared__ __align__(8) uint64_t conv_empty_bar[kMaxStages];  // decoded slot free (NVFP4)
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t accf_bar[kMaxAcc];
  __shared__ __align__(8) uint64_t acce_bar[kMaxAcc];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int c = 0; c < p.conv_stages; ++c) {
      mbar_init(&conv_bar[c], kConvThreads);
      mbar_init(&conv_empty_bar[c], 1);
    }
    for (int a = 0; a < p.acc_bufs; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], kEpiThreads);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmB64);
    tma_prefetch_desc(&tmB128);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the work items, tokens and h come from earlier work on the stream

  constexpr bool kConv = kFmt != kFmtBf16;    // weights decoded into tensor memory
  constexpr bool kFp8 = kFmt == kFmtFp8;
  constexpr uint32_t kPB = kFp8 ? kP8TileBytes : kPTileBytes;  // raw weight tile bytes (kConv)
  const uint32_t tmem_base = tmem_slot;
  const int n_items = *p.n_items;
  const int kblocks = p.K / BK;
  constexpr int nA = 2;                       // weight tiles per item
  constexpr int kItemRows = kGLU ? BM : 2 * BM;  // weight rows an item covers
  constexpr int kRow1 = kGLU ? 0 : BM;          // row offset of tile 1 (up tile / second down tile)
  long long fills = 0;  // TMA stage fills issued (thread 0 only)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int4 item = work_item(p.table, p.tile_expert, p.wt, it);
        const int a_row = item.x * p.Nw + item.y * kItemRows;
        const int nbox = (item.w + TOK_BOX - 1) / TOK_BOX;
        const uint32_t bytes = (kConv ? kPB : kATileBytes) * nA + static_cast<uint32_t>(nbox) * kTokBoxBytes;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, p.wait_spins, kWaitNs, abort, kSleepSlotNs)) {
            if (!*abort) fail(p, abort, 1);
            ok = false;
            break;
          }
          uint8_t* st = smem + static_cast<size_t>(stage) * p.stage_bytes;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          if (kConv) {
            // raw codes of one 64-element K slice: 32 bytes (e2m1) or 64 bytes (e4m3) per row
            const int x0 = kb * static_cast<int>(kPB / BM);
            tma_load_2d(st + p.p_offset, &tmA0, x0, a_row, &full_bar[stage]);
            tma_load_2d(st + p.p_offset + kPB, &tmA1, x0, a_row + kRow1, &full_bar[stage]);
          } else {
            tma_load_2d(st, &tmA0, kb * BK, a_row, &full_bar[stage]);
            tma_load_2d(st + kATileBytes, &tmA1, kb * BK, a_row + kRow1, &full_bar[stage]);
          }
          // token rows in boxes of 128, 64 and 16 rows (fewest copies); the
          // stacked boxes form one 128-byte-swizzled K-major tile
          uint8_t* sb = st + p.b_offset;
          int row = item.z, left = nbox * TOK_BOX;
          for (; left >= 128; left -= 128, row += 128, sb += 128 * BK * 2)
            tma_load_2d(sb, &tmB128, kb * BK, row, &full_bar[stage]);
          if (left >= 64) {
            tma_load_2d(sb, &tmB64, kb * BK, row, &full_bar[stage]);
            left -= 64;
            row += 64;
            sb += 64 * BK * 2;
          }
          for (; left > 0; left -= TOK_BOX, row += TOK_BOX, sb += kTokBoxBytes)
            tma_load_2d(sb, &tmB, kb * BK, row, &full_bar[stage]);
          ++fills;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0, cstage = 0;
      uint32_t phase = 0, acc_phase = 0, cphase = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int4 item = work_item(p.table, p.tile_expert, p.wt, it);
        const int n_mma = (item.w + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
        if (!mbar_wait_bounded(&acce_bar[acc], acc_phase ^ 1u, p.wait_spins, kWaitNs, abort)) {
          if (!*abort) fail(p, abort, 2);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * p.acc_cols);
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t st_addr = smem_u32(smem + static_cast<size_t>(stage) * p.stage_bytes);
          // one shared-memory descriptor per operand; a 16-wide K step (32 bytes) adds 2 to
          // the start address field (bits 0-13, bytes >> 4), which never carries out of it
          const uint64_t b0 = sdesc_kmajor_sw128(st_addr + p.b_offset);
          if constexpr (kConv) {
            // NVFP4 / FP8: the decoded slot is ready only after its raw stage landed. Slot
            // columns: tile 0 [0, 32), tile 1 [32, 64), 8 per 16-wide K step.
            if (!mbar_wait_bounded(&conv_bar[cstage], cphase, p.wait_spins, kWaitNs, abort)) {
              if (!*abort) fail(p, abort, 3);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t ta = tmem_base + p.a_col + static_cast<uint32_t>(cstage * kConvCols);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
              mma_bf16_ts(d0, ta + k * 8, b0 + 2 * k, idesc, accum);
              mma_bf16_ts(d1, ta + kConvCols / 2 + k * 8, b0 + 2 * k, idesc, accum);
            }
            mma_commit(&conv_empty_bar[cstage]);
            if (++cstage == p.conv_stages) {
              cstage = 0;
              cphase ^= 1u;
            }
          } else {
            if (!mbar_wait_bounded(&full_bar[stage], phase, p.wait_spins, kWaitNs, abort)) {
              if (!*abort) fail(p, abort, 3);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a0 = sdesc_kmajor_sw128(st_addr), a1 = sdesc_kmajor_sw128(st_addr + kATileBytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
              mma_bf16_ss(d0, a0 + 2 * k, b0 + 2 * k, idesc, accum);
              mma_bf16_ss(d1, a1 + 2 * k, b0 + 2 * k, idesc, accum);
            }
          }
          mma_commit(&empty_bar[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&accf_bar[acc]);
        if (++acc == p.acc_bufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const int eg = (warp - 2) >> 2;  // epilogue warpgroup: 16-token chunks eg, eg + 2, ...
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int4 item = work_item(p.table, p.tile_expert, p.wt, it);
      // tcgen05.ld is warp-collective: the whole warp proceeds or stops together
      const bool ok = __all_sync(
          0xffffffffu, mbar_wait_bounded(&accf_bar[acc], acc_phase, p.wait_spins, kWaitNs, abort, kSleepItemNs));
      if (!ok) {
        if (lane == 0 && !*abort) fail(p, abort, 4);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * p.acc_cols);
      // debug build: the item's rows and expert lie inside the buffers
      const bool item_ok = dcheck(item.x >= 0 && item.x < p.E && item.z >= 0 && item.w >= 0 && item.w <= p.n_max &&
                                      static_cast<int64_t>(item.z) + item.w <= p.R,
                                  p.status);
      const int col0 = item.y * kItemRows + r;       // output column of accumulator 0
      const int col1 = col0 + kRow1;                 // ... of accumulator 1 (GEMM2)
      const bool valid0 = col0 < p.Nw, valid1 = col1 < p.Nw;
      const int ntok = item_ok ? item.w : 0;
      const float s0 = p.ts0 && item_ok ? p.ts0[item.x] : 1.0f;
      const float s1 = p.ts1 && item_ok ? p.ts1[item.x] : s0;
      // 16-token chunks eg*16, eg*16 + 32, ...: the TMEM loads of the next chunk
      // are in flight while this one is computed and stored, and the
      // accumulator is handed back to the MMA as soon as the last chunk's loads
      // have landed (its math and stores overlap the next item's MMAs).
      auto load_chunk = [&](int c, uint32_t (&gg)[16], uint32_t (&uu)[16]) {
        tmem_ld_32x32b_x16(tb + c, gg);
        tmem_ld_32x32b_x16(tb + p.n_max + c, uu);
      };
      auto store_chunk = [&](int c, const uint32_t (&gg)[16], const uint32_t (&uu)[16]) {
        if (kGLU) {
          if (valid0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tok = c + j;
              if (tok < ntok) {
                const float gv = __uint_as_float(gg[j]) * s0;
                const float uv = __uint_as_float(uu[j]) * s1;
                // silu(g) = g / (1 + e^-g); h is rounded to bf16 right after, so the
                // fast exponential and division (relative error ~1e-7) do not show
                const float silu = __fdividef(gv, 1.0f + __expf(-gv));
                p.h_out[static_cast<size_t>(item.z + tok) * p.Nw + col0] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(silu * uv));
              }
            }
          }
        } else if (p.y_f32) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c + j;
            if (tok < ntok) {
              float* yrow = p.y_f32 + static_cast<size_t>(item.z + tok) * p.Nw;
              if (valid0) yrow[col0] = __uint_as_float(gg[j]) * s0;
              if (valid1) yrow[col1] = __uint_as_float(uu[j]) * s0;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c + j;
            if (tok < ntok) {
              uint16_t* yrow = p.y_out + static_cast<size_t>(item.z + tok) * p.Nw;
              if (valid0) yrow[col0] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(gg[j]) * s0));
              if (valid1) yrow[col1] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(uu[j]) * s0));
            }
          }
        }
      };
      uint32_t ga[16], ua[16], gb[16], ub[16];
      bool released = false;
      auto next_or_release = [&](int cn, uint32_t (&gg)[16], uint32_t (&uu)[16]) {
        if (cn < ntok) {
          load_chunk(cn, gg, uu);
        } else {
          tc_fence_before();
          mbar_arrive(&acce_bar[acc]);
          released = true;
        }
      };
      int c = eg * 16;
      if (c < ntok) load_chunk(c, ga, ua);
      while (c < ntok) {
        tmem_ld_wait();
        next_or_release(c + 32, gb, ub);
        store_chunk(c, ga, ua);
        c += 32;
        if (c >= ntok) break;
        tmem_ld_wait();
        next_or_release(c + 32, ga, ua);
        store_chunk(c, gb, ub);
        c += 32;
      }
      if (!released) {
        tc_fence_before();
        mbar_arrive(&acce_bar[acc]);
      }
      if (++acc == p.acc_bufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (kConv) {
    // ------------------------------------------------------------ NVFP4 / FP8 converters
    // Warp 10 + 4t + j decodes weight tile t (gate/up, or the two down tiles)
    // for the 32 rows of the TMEM lane quarter it may access (warp % 4); one
    // thread per row. Scales are read from global memory one group of four
    // K slices ahead, so the load latency hides behind decoding:
    //   NVFP4: 4 e4m3 block scales per slice per row, 16 bytes (four slices) a load;
    //   FP8: one fp32 scale per 128 x 128 block, uniform over the tile (tiles
    //   start on 128-row boundaries) and shared by two 64-wide slices.
    const int t = (warp - kConvBase / 32) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int row_off = t ? kRow1 : 0;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + p.a_col +
                            static_cast<uint32_t>(t * (kConvCols / 2));  // this tile's 32 columns of a slot
    int stage = 0, cstage = 0;
    uint32_t phase = 0, cphase = 0;
    // scale group g of `item` (expert -1: none): slices 4g .. 4g+3
    auto load_group = [&](const int4& item, int g) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (item.x < 0) return v;
      if (!dcheck(item.x < p.E, p.status)) return v;
      if constexpr (kFp8) {
        const int nbr = p.Nw / BM, kbr = p.K / BM;  // 128-blocks per expert: rows, K
        const int br = (item.y * kItemRows + row_off) / BM;
        // padding rows past the expert (ragged last down tile) get scale 0
        if (br < nbr) {
          const float* f = (t ? p.fs1 : p.fs0) + (static_cast<int64_t>(item.x) * nbr + br) * kbr;
          const int k0 = 2 * g;  // 128-wide K blocks covered by slices 4g .. 4g+3
          v.x = __float_as_uint(__ldg(f + k0));
          if (k0 + 1 < kbr) v.y = __float_as_uint(__ldg(f + k0 + 1));
        }
      } else {
        const int sf_ld = p.K / 16;  // bytes of block scales per weight row
        const int64_t rows_total = static_cast<int64_t>(p.E) * p.Nw;
        const int64_t row = static_cast<int64_t>(item.x) * p.Nw + item.y * kItemRows + row_off + r;
        // padding rows past the last expert decode to zero
        if (row < rows_total)
          v = __ldg(reinterpret_cast<const uint4*>((t ? p.sf1 : p.sf0) + row * sf_ld + g * 16));
      }
      return v;
    };
    // the item's schedule entry is looked up once per item (the next one a group ahead)
    auto item_at = [&](int it) { return it < n_items ? work_item(p.table, p.tile_expert, p.wt, it) : make_int4(-1, 0, 0, 0); };
    int4 item = item_at(blockIdx.x);
    uint4 cur = make_uint4(0, 0, 0, 0), nxt = load_group(item, 0);
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 next_item = item_at(it + gridDim.x);
      for (int kb = 0; kb < kblocks; ++kb) {
        if ((kb & 3) == 0) {
          cur = nxt;
          nxt = kb + 4 < kblocks ? load_group(item, (kb >> 2) + 1) : load_group(next_item, 0);
        }
        const uint8_t* packed = smem + static_cast<size_t>(stage) * p.stage_bytes + p.p_offset + t * kPB;
        const int g = kb & 3;
        // tcgen05.st is warp-collective: the whole warp proceeds or stops together
        const bool ready = __all_sync(
            0xffffffffu,
            mbar_wait_bounded(&full_bar[stage], phase, p.wait_spins, kWaitNs, abort, kSleepSlotNs) &&
                mbar_wait_bounded(&conv_empty_bar[cstage], cphase ^ 1u, p.wait_spins, kWaitNs, abort, kSleepSlotNs));
        if (!ready) {
          if (lane == 0 && !*abort) fail(p, abort, 5);
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this slot have completed
        // the row's two 32-element halves, each stored as soon as it is decoded
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          uint32_t v[16];
          if constexpr (kFp8) {
            decode_half_fp8(packed, r, hk, __uint_as_float(g < 2 ? cur.x : cur.y), v);
          } else {
            decode_half(packed, r, hk, g == 0 ? cur.x : g == 1 ? cur.y : g == 2 ? cur.z : cur.w, v);
          }
          tmem_st_32x32b_x16(t_lane + static_cast<uint32_t>(cstage * kConvCols + hk * 16), v);
        }
        tmem_st_wait();
        fence_proxy_async_smem();  // the packed tile's reads complete before TMA may refill the stage
        tc_fence_before();
        mbar_arrive(&conv_bar[cstage]);
        if (++cstage == p.conv_stages) {
          cstage = 0;
          cphase ^= 1u;
        }
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      item = next_item;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort) {
    // Every role has stopped. Let the copies and MMAs this CTA issued land
    // before its shared memory and TMEM are released.
    if (threadIdx.x == 0) {
      for (int s = 0; s < p.stages; ++s) {
        if (fills > s) {
          const long long f = s + static_cast<long long>(p.stages) * ((fills - 1 - s) / p.stages);
          mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((f / p.stages) & 1), 1ll << 40, kDrainNs, nullptr);
        }
      }
    }
    if (warp == 1 && lane == 0) {
      mma_commit(&drain_bar);
      mbar_wait_bounded(&drain_bar, 0, 1ll << 40, kDrainNs, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// The work schedule from the expert offsets (build_schedule): one thread per expert (E <= 256).
__global__ void __launch_bounds__(256) schedule_kernel(const int32_t* __restrict__ offsets, int E, ScheduleArgs s,
                                                       int32_t* status) {
  __shared__ int warp_sums[8];
  pdl_launch_dependents();
  pdl_wait();
  build_schedule(offsets, E, s, status, warp_sums);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 2-D bf16 tensor [outer][inner] (inner contiguous), box [box_outer][64],
// 128-byte swizzle, zero fill out of bounds.
int encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

// 2-D byte tensor [outer][inner_bytes] of weight codes, box [128][box_bytes]
// (one 64-element K slice of 128 weight rows: 32 bytes of e2m1, 64 of e4m3),
// no swizzle.
int encode_packed_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t outer, uint32_t box_bytes) {
  auto fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[2] = {inner_bytes, outer};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {box_bytes, static_cast<cuuint32_t>(BM)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

struct StageShape {
  int stages, acc_bufs, acc_cols, conv_stages;
  uint32_t stage_bytes, b_offset, p_offset, a_col;
  size_t smem;
};

StageShape stage_shape(bool glu, int fmt, int n_max) {
  StageShape s;
  (void)glu;
  const int budget = kSmemLimit - 1024 - 512;  // alignment slack + static barriers
  const uint32_t b_bytes = static_cast<uint32_t>(n_max) * BK * 2;
  s.acc_cols = 2 * n_max;
  if (fmt != kFmtBf16) {
    // ring stage: token rows, then the two raw weight tiles. TMEM: the
    // accumulators, then 2-4 decoded slots (at least 3 where that leaves one
    // accumulator buffer); n_max <= 192 keeps two slots.
    const uint32_t pb = fmt == kFmtFp8 ? kP8TileBytes : kPTileBytes;
    s.b_offset = 0;
    s.p_offset = b_bytes;
    s.stage_bytes = (b_bytes + 2 * pb + 1023u) & ~1023u;
    s.acc_bufs = std::max(1, std::min(kMaxAcc, (static_cast<int>(kTmemCols) - 3 * kConvCols) / s.acc_cols));
    s.a_col = static_cast<uint32_t>(s.acc_bufs * s.acc_cols);
    s.conv_stages = std::min(kMaxConv, (static_cast<int>(kTmemCols) - static_cast<int>(s.a_col)) / kConvCols);
  } else {
    s.b_offset = 2 * kATileBytes;
    s.p_offset = s.b_offset + b_bytes;
    s.stage_bytes = (s.p_offset + 1023u) & ~1023u;
    s.acc_bufs = std::min(kMaxAcc, static_cast<int>(kTmemCols) / s.acc_cols);
    s.a_col = 0;
    s.conv_stages = 0;
  }
  s.stages = std::min(kMaxStages, budget / static_cast<int>(s.stage_bytes));
  s.smem = 1024 + static_cast<size_t>(s.stages) * s.stage_bytes;
  return s;
}

template <bool kGLU, int kFmt>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap (&b)[3], GemmArgs args,
                        int n_max, int grid, cudaStream_t stream) {
  const StageShape s = stage_shape(kGLU, kFmt, n_max);
  if (kFmt != kFmtBf16 && s.conv_stages < 2) return cudaErrorInvalidValue;  // n_max above 192
  args.stages = s.stages;
  args.acc_bufs = s.acc_bufs;
  args.acc_cols = s.acc_cols;
  args.stage_bytes = s.stage_bytes;
  args.b_offset = s.b_offset;
  args.p_offset = s.p_offset;
  args.a_col = s.a_col;
  args.conv_stages = s.conv_stages;
  args.n_max = n_max;
  cudaError_t err = cudaFuncSetAttribute(expert_gemm_kernel<kGLU, kFmt>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s.smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(expert_gemm_kernel<kGLU, kFmt>, dim3(grid), dim3(threads_for(kFmt)), s.smem, stream, a0, a1, b[0],
                    b[1], b[2], args);
}

}  // namespace

ExpertPlan plan_experts(int T, int d, int E, int top_k, int inter, bool decoded) {
  ExpertPlan p;
  // Token tile: a quarter above the mean tokens per expert, at least 64 and at
  // most 256 (the MMA's largest N; 192 with NVFP4 or FP8 weights, whose decoded tiles
  // share tensor memory with the accumulators), never above the batch (an
  // expert sees a token at most once). Smaller tiles leave shared memory for
  // more pipeline stages; experts above the tile are split into near-equal tiles.
  const int64_t R = static_cast<int64_t>(T) * top_k;
  const int64_t mean = (R + E - 1) / std::max(E, 1);
  int64_t n = ((mean + mean / 4 + 15) / 16) * 16;
  n = std::max<int64_t>(64, std::min<int64_t>(decoded ? 192 : 256, n));
  const int tok = ((std::max(T, 1) + 15) / 16) * 16;
  p.n_max = static_cast<int>(std::min<int64_t>(n, tok));
  p.max_tiles = static_cast<int>(E + (R + p.n_max - 1) / p.n_max);
  p.wtiles1 = (inter + BM - 1) / BM;
  p.wtiles2 = (d + 2 * BM - 1) / (2 * BM);
  return p;
}

ScheduleArgs schedule_args(const ExpertPlan& plan, const ExpertBuffers& buf, int R) {
  ScheduleArgs s;
  s.n_max = plan.n_max;
  s.wt1 = plan.wtiles1;
  s.wt2 = plan.wtiles2;
  s.R = R;
  s.table = buf.table;
  s.tile_expert = buf.tile_expert;
  s.max_tiles = plan.max_tiles;
  s.n_items = buf.n_items;
  return s;
}

cudaError_t launch_expert_ffn(const ExpertPlan& plan, const ExpertBuffers& buf, const ExpertWeightsDev& w, int T,
                              int d, int E, int top_k, int inter, int num_sms, long long wait_spins,
                              cudaStream_t stream, int* cu_error, cudaEvent_t after_gemm1, bool items_ready) {
  *cu_error = 0;
  const int R = T * top_k;
  const int fmt = w.wfmt;
  if (fmt != MOE_W_BF16 && fmt != MOE_W_NVFP4 && fmt != MOE_W_FP8) return cudaErrorInvalidValue;
  if (fmt == MOE_W_NVFP4 && ((d % 256) || (inter % 256))) return cudaErrorNotSupported;
  if (fmt == MOE_W_FP8 && ((d % 128) || (inter % 128))) return cudaErrorNotSupported;
  cudaError_t err = cudaSuccess;
  if (!items_ready) {  // otherwise the permutation's plan kernel built them
    err = launch_pdl(schedule_kernel, dim3(1), dim3(256), 0, stream, buf.offsets, E, schedule_args(plan, buf, R),
                     buf.status);
    if (err != cudaSuccess) return err;
  }

  CUtensorMap tg, tu, td, tx[3], th[3];
  int rc = 0;
  if (fmt == MOE_W_NVFP4) {
    rc |= encode_packed_2d(&tg, w.gate, d / 2, static_cast<uint64_t>(E) * inter, BK / 2);
    rc |= encode_packed_2d(&tu, w.up, d / 2, static_cast<uint64_t>(E) * inter, BK / 2);
    rc |= encode_packed_2d(&td, w.down, inter / 2, static_cast<uint64_t>(E) * d, BK / 2);
  } else if (fmt == MOE_W_FP8) {
    rc |= encode_packed_2d(&tg, w.gate, d, static_cast<uint64_t>(E) * inter, BK);
    rc |= encode_packed_2d(&tu, w.up, d, static_cast<uint64_t>(E) * inter, BK);
    rc |= encode_packed_2d(&td, w.down, inter, static_cast<uint64_t>(E) * d, BK);
  } else {
    rc |= encode_bf16_2d(&tg, w.gate, d, static_cast<uint64_t>(E) * inter, BM);
    rc |= encode_bf16_2d(&tu, w.up, d, static_cast<uint64_t>(E) * inter, BM);
    rc |= encode_bf16_2d(&td, w.down, inter, static_cast<uint64_t>(E) * d, BM);
  }
  const uint32_t boxes[3] = {TOK_BOX, 64, 128};
  for (int i = 0; i < 3; ++i) {
    rc |= encode_bf16_2d(&tx[i], buf.x_perm, d, R, boxes[i]);
    rc |= encode_bf16_2d(&th[i], buf.h, inter, R, boxes[i]);
  }
  if (rc) {
    *cu_error = rc;
    return cudaErrorInvalidValue;
  }
  GemmArgs a1{};
  a1.table = buf.table;
  a1.tile_expert = buf.tile_expert;
  a1.wt = plan.wtiles1;
  a1.n_items = buf.n_items;
  a1.K = d;
  a1.Nw = inter;
  a1.E = E;
  a1.R = R;
  a1.h_out = buf.h;
  a1.status = buf.status;
  a1.timeout_where = buf.timeout_where;
  a1.wait_spins = wait_spins;
  if (fmt == MOE_W_NVFP4) {
    a1.ts0 = w.gate_ts;
    a1.ts1 = w.up_ts;
    a1.sf0 = static_cast<const uint8_t*>(w.gate_sf);
    a1.sf1 = static_cast<const uint8_t*>(w.up_sf);
    err = launch_gemm<true, kFmtNvfp4>(tg, tu, tx, a1, plan.n_max, num_sms, stream);
  } else if (fmt == MOE_W_FP8) {
    a1.fs0 = static_cast<const float*>(w.gate_sf);
    a1.fs1 = static_cast<const float*>(w.up_sf);
    err = launch_gemm<true, kFmtFp8>(tg, tu, tx, a1, plan.n_max, num_sms, stream);
  } else {
    err = launch_gemm<true, kFmtBf16>(tg, tu, tx, a1, plan.n_max, num_sms, stream);
  }
  if (err != cudaSuccess) return err;
  if (after_gemm1 && (err = cudaEventRecord(after_gemm1, stream)) != cudaSuccess) return err;
  GemmArgs a2{};
  a2.table = buf.table;
  a2.tile_expert = buf.tile_expert;
  a2.wt = plan.wtiles2;
  a2.n_items = buf.n_items + 1;
  a2.K = inter;
  a2.Nw = d;
  a2.E = E;
  a2.R = R;
  a2.y_out = buf.y;
  a2.y_f32 = buf.y_f32;
  a2.status = buf.status;
  a2.timeout_where = buf.timeout_where;
  a2.wait_spins = wait_spins;
  if (fmt == MOE_W_NVFP4) {
    a2.ts0 = w.down_ts;
    a2.sf0 = static_cast<const uint8_t*>(w.down_sf);
    a2.sf1 = a2.sf0;
    return launch_gemm<false, kFmtNvfp4>(td, td, th, a2, plan.n_max, num_sms, stream);
  }
  if (fmt == MOE_W_FP8) {
    a2.fs0 = static_cast<const float*>(w.down_sf);
    a2.fs1 = a2.fs0;
    return launch_gemm<false, kFmtFp8>(td, td, th, a2, plan.n_max, num_sms, stream);
  }
  return launch_gemm<false, kFmtBf16>(td, td, th, a2, plan.n_max, num_sms, stream);
}

}  // namespace beammoe
