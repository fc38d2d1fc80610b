// Allocation-free variant of the permutation step (moe_permute_noalloc).
//
// Some callers cannot allocate device memory at all: code that runs while a
// CUDA graph is being captured, a serving loop that must never call
// cudaMalloc (it can synchronise the device and stall other streams), or a
// plugin inside a host framework that owns every device buffer and offers no
// allocator hook. moe_permute needs a caller-provided workspace for its
// scratch; this variant keeps that scratch in a fixed, file-scope device
// array instead, so the caller passes only inputs and outputs.
//
// The array below is a static device allocation of kScratchBytes (about
// 1 MiB) that every GPU which loads this library holds until the process
// exits. Its contents persist from call to call and are shared by all calls,
// so each call clears what must start at zero (its status word and, inside
// the permutation launch, the bitmap), and calls that overlap on the GPU race
// on it (run them on one stream).
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// Largest permutation the static scratch covers.
constexpr int kNoAllocMaxT = 16384;
constexpr int kNoAllocMaxE = 256;
constexpr size_t kNoAllocWords = static_cast<size_t>(kNoAllocMaxE) * ((kNoAllocMaxT + 31) / 32);
// [0, 256): status word; then the bitmap words; then the per-word prefix counts
constexpr size_t kScratchBytes = 256 + 2 * kNoAllocWords * sizeof(uint32_t);

static __device__ __align__(256) uint8_t g_permute_scratch[kScratchBytes];

// Host code cannot use the array's name as a device address (it names a
// host-side stand-in), so its device address is looked up per device and
// kept once the lookup has succeeded; a failed lookup is tried again on the
// next call.
constexpr int kMaxDevices = 64;
struct DeviceScratch {
  std::mutex lock;
  std::atomic<void*> ptr{nullptr};
};
DeviceScratch g_scratch[kMaxDevices];

void* scratch_address(int dev) {
  DeviceScratch& s = g_scratch[dev];
  void* p = s.ptr.load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> guard(s.lock);
  p = s.ptr.load(std::memory_order_relaxed);
  if (!p && cudaGetSymbolAddress(&p, g_permute_scratch) == cudaSuccess && p)
    s.ptr.store(p, std::memory_order_release);
  return p;
}

moe_status_t check_permute_dims(const moe_dims_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->d <= 0 || d->E <= 0 || d->n_groups <= 0 || d->topk_groups <= 0 || d->top_k <= 0 ||
      d->inter <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->E % d->n_groups != 0 || d->topk_groups > d->n_groups || d->top_k > d->topk_groups * (d->E / d->n_groups))
    return MOE_ERR_INVALID_ARG;
  if (d->d % 64 || d->d > 16384 || d->inter % 64 || d->inter > 16384 || d->n_groups > 32 || d->top_k > 32)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_permute_noalloc(const moe_dims_t* dims, const moe_bf16_t* x, const int32_t* topk_idx,
                                            int32_t* counts, int32_t* offsets, int32_t* row_token,
                                            int32_t* inv_row, moe_bf16_t* x_perm, int32_t* device_status,
                                            void* stream) {
  moe_status_t st = check_permute_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T > kNoAllocMaxT || dims->E > kNoAllocMaxE) return MOE_ERR_SCRATCH_LIMIT;
  if (dims->T == 0) {  // nothing to permute; the caller's status word still reports this call
    if (device_status &&
        cudaMemsetAsync(device_status, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!aligned16(x) || !topk_idx || !counts || !offsets || !row_token || !inv_row || !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MOE_ERR_CUDA;
  if (dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* scratch = scratch_address(dev);
  if (!scratch) return MOE_ERR_CUDA;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  int32_t* status = reinterpret_cast<int32_t*>(base);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(base + 256);
  int32_t* word_prefix = reinterpret_cast<int32_t*>(base + 256 + kNoAllocWords * sizeof(uint32_t));

  if (cudaMemsetAsync(status, 0, sizeof(int32_t), cs) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t e = beammoe::launch_permute(x, topk_idx, dims->T, dims->d, dims->E, dims->top_k, bitmap,
                                                word_prefix, counts, offsets, row_token, inv_row, x_perm, status, cs);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (device_status &&
      cudaMemcpyAsync(device_status, status, sizeof(int32_t), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
