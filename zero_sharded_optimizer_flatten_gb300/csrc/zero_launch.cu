// Kernel dispatch and grid sizing.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "zero_kernels.cuh"

namespace zero {

extern template int launch_typed<__half>(Kind, const LaunchArgs&, cudaStream_t);
extern template int launch_typed<__nv_bfloat16>(Kind, const LaunchArgs&, cudaStream_t);

int grid_for(const void* fn, int64_t n_tiles) {
  constexpr int64_t kMaxGrid = 0x7fffffff;  // grid.x limit; CTAs stride beyond it
  if (ZERO_GRID_MULT == 0) return static_cast<int>(n_tiles < kMaxGrid ? n_tiles : kMaxGrid);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int slots = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({fn, dev});
    if (it != cache.end()) {
      slots = it->second;
    } else {
      int per_sm = 0, sms = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0) != cudaSuccess)
        return -1;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
      slots = (per_sm > 0 ? per_sm : 1) * sms * ZERO_GRID_MULT;
      cache[{fn, dev}] = slots;
    }
  }
  return static_cast<int>(n_tiles < slots ? n_tiles : slots);
}

int launch_kernel(Kind kind, zero_dtype dtype, const LaunchArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == ZERO_BF16) return launch_typed<__nv_bfloat16>(kind, a, s);
  return launch_typed<__half>(kind, a, s);
}

}  // namespace zero
