// zero_step_amp_noalloc: the mixed-precision step for callers that cannot
// allocate device memory.  Its scratch space is a fixed array compiled into
// the library instead of a caller-provided workspace; see include/zero.h.
#include <cuda_runtime.h>
#include <inttypes.h>

#include <mutex>

#include "zero_capi_util.h"
#include "zero_internal.h"

namespace {

// The library's own scratch for zero_step_amp_noalloc: 2 MiB, which holds the
// 8 KB workspace head (decision-record copies, the decision kernel's sums)
// plus 130,560 per-tile sums of squares of 16 bytes each (groups of up to
// 267,386,880 owned elements per step).  It exists once on every GPU that
// loads the library and stays there until the process exits.
constexpr int64_t kNoAllocScratchBytes = INT64_C(2) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name only stands for the symbol, so the address is looked up
// once per device, with that device current, and cached.  Under lazy module
// loading the first lookup on a device also loads the module and commits the
// array; the cached address stays valid for the life of the device's
// context (a cudaDeviceReset would invalidate it).
zero_status scratch_on_current_device(const char* fn, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return zero::fail(ZERO_ERR_CUDA, "%s: cudaGetDevice: %s", fn, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return zero::fail(ZERO_ERR_UNSUPPORTED, "%s: device %d is beyond the %d this entry point tracks",
                      fn, dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return zero::fail(ZERO_ERR_CUDA, "%s: cudaGetSymbolAddress of the fixed scratch failed: %s", fn,
                        cudaGetErrorString(e));
    g_dev_ptr[dev] = p;
  }
  *out = g_dev_ptr[dev];
  return ZERO_OK;
}

}  // namespace

extern "C" zero_status zero_step_amp_noalloc(const zero_plan* plan, const void* const* grads,
                                             zero_dtype dtype, zero_reduce_op op,
                                             float* const* grad_shards, float* const* master,
                                             float* const* m, float* const* v, void* full_flat16,
                                             void* const* out16_shard,
                                             const zero_adamw_hparams* hp,
                                             const zero_amp_config* cfg, void* d_state,
                                             uint64_t rank_mask, int64_t bucket_elems,
                                             void* stream) {
  const char* fn = "zero_step_amp_noalloc";
  int64_t need = 0;
  zero_status st = zero_amp_workspace_bytes(plan, rank_mask, bucket_elems, &need);
  if (st != ZERO_OK) return st;
  if (need > kNoAllocScratchBytes)
    return zero::fail(ZERO_ERR_INVALID,
                      "%s: this step needs %" PRId64 " bytes of scratch but the library's fixed "
                      "scratch holds %" PRId64 " (at most %" PRId64 " tiles of 2048 elements); "
                      "use zero_step_amp with a caller-allocated workspace",
                      fn, need, kNoAllocScratchBytes,
                      (kNoAllocScratchBytes - zero::kAmpHeadBytes) /
                          static_cast<int64_t>(sizeof(zero::NormPartial)));
  void* scratch = nullptr;
  st = scratch_on_current_device(fn, &scratch);
  if (st != ZERO_OK) return st;
  // Every byte of the scratch that this step reads is written earlier in the
  // same step (each tile's partial sum, the beta powers and the arrival
  // counter by the reduction; the per-CTA sums and the decision record by the
  // decision kernel), so nothing has to be cleared between calls.
  return zero_step_amp(plan, grads, dtype, op, grad_shards, master, m, v, full_flat16,
                       out16_shard, hp, cfg, d_state, scratch, kNoAllocScratchBytes, rank_mask,
                       bucket_elems, stream);
}
