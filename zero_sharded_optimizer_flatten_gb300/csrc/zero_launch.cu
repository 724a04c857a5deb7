// Kernel dispatch and grid sizing.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "zero_kernels.cuh"
#include "zero_kernels_tma.cuh"

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

// The decision of the mixed-precision step (one CTA): sum the per-tile
// partials in a fixed order, then update the loss-scale state and form the
// step's coefficient and AdamW constants (binary64, each rounded once).
constexpr int kFinalizeThreads = 1024;

__device__ void amp_decide(zero_amp_state& x, double sumsq, const AmpParams& p) {
  const double S = x.scale;
  x.norm = sqrt(sumsq) / S;
  if (!isfinite(sumsq)) {
    x.overflow = 1;
    x.skipped += 1;
    x.good_steps = 0;
    x.coef = 0.0f;
    if (x.hysteresis_left > 1) {
      x.hysteresis_left -= 1;
    } else {
      const double half = S / 2.0;
      x.scale = half > p.cfg.min_scale ? half : p.cfg.min_scale;
    }
    return;
  }
  double clip = 1.0;
  if (p.cfg.max_norm > 0.0) {
    const double q = p.cfg.max_norm / (x.norm + 1e-6);
    if (q < 1.0) clip = q;
  }
  x.coef = static_cast<float>(clip / S);
  const int64_t t = x.step + 1;
  const zero_adamw_hparams& h = p.hp;
  x.sc[0] = static_cast<float>(1.0 - h.lr * h.weight_decay);
  x.sc[1] = static_cast<float>(h.beta1);
  x.sc[2] = static_cast<float>(h.beta2);
  x.sc[3] = static_cast<float>(1.0 - h.beta1);
  x.sc[4] = static_cast<float>(1.0 - h.beta2);
  x.sc[5] = static_cast<float>(h.lr / (1.0 - pow(h.beta1, static_cast<double>(t))));
  x.sc[6] = static_cast<float>(sqrt(1.0 - pow(h.beta2, static_cast<double>(t))));
  x.sc[7] = static_cast<float>(h.eps);
  x.overflow = 0;
  x.step = t;
  x.good_steps += 1;
  if (p.cfg.window > 0 && x.good_steps >= p.cfg.window) {
    x.scale = S * 2.0;
    x.good_steps = 0;
    x.hysteresis_left = p.cfg.hysteresis;
  }
}

__global__ void __launch_bounds__(kFinalizeThreads) k_amp_finalize(const double* partials,
                                                                   int64_t n,
                                                                   zero_amp_state* st,
                                                                   AmpBcast* bcast,
                                                                   const AmpParams p) {
  // four independent running sums per thread (fixed assignment), then the
  // block in a fixed order
  double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
  constexpr int64_t kStride = 4 * kFinalizeThreads;
  int64_t i = threadIdx.x;
  for (; i + 3 * kFinalizeThreads < n; i += kStride) {
    s0 += __ldcg(partials + i);
    s1 += __ldcg(partials + i + kFinalizeThreads);
    s2 += __ldcg(partials + i + 2 * kFinalizeThreads);
    s3 += __ldcg(partials + i + 3 * kFinalizeThreads);
  }
  for (; i < n; i += kFinalizeThreads) s0 += __ldcg(partials + i);
  const double sumsq = block_sum<kFinalizeThreads>((s0 + s1) + (s2 + s3));
  __shared__ AmpBcast rec;
  if (threadIdx.x == 0) {
    zero_amp_state x = *st;
    amp_decide(x, sumsq, p);
    *st = x;
    AmpBcast b = {};
    b.overflow = x.overflow;
    b.coef = x.coef;
    for (int k = 0; k < 8; ++k) b.sc[k] = x.sc[k];
    rec = b;
  }
  __syncthreads();
  // the decision record to its kAmpCopies places, one thread each
  if (threadIdx.x < kAmpCopies) bcast[threadIdx.x] = rec;
}

__global__ void k_amp_init(zero_amp_state* st, const zero_amp_state v) { *st = v; }

int launch_amp_finalize(const double* partials, int64_t n_tiles, zero_amp_state* state,
                        AmpBcast* bcast, const AmpParams& p, void* stream) {
  k_amp_finalize<<<1, kFinalizeThreads, 0, static_cast<cudaStream_t>(stream)>>>(partials, n_tiles,
                                                                               state, bcast, p);
  return static_cast<int>(cudaGetLastError());
}

int launch_amp_init(zero_amp_state* state, const zero_amp_state& init, void* stream) {
  k_amp_init<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(state, init);
  return static_cast<int>(cudaGetLastError());
}

int tma_grid(const void* fn, int smem_bytes, int64_t n_tiles) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({fn, dev});
  if (it == cache.end()) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
        cudaSuccess)
      return -1;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem_bytes) !=
        cudaSuccess)
      return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return -1;
    it = cache.emplace(std::make_pair(fn, dev), (per_sm > 0 ? per_sm : 1) * sms).first;
  }
  return static_cast<int>(n_tiles < it->second ? n_tiles : it->second);
}

// The device error word: set by a kernel whose bounded wait gave up.
static __device__ int g_device_error;

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::mutex mu;
  static int* ptr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int*>(p);
  }
  return ptr[dev];
}

int take_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof v, 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return 0;
  if (v) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                s) == cudaSuccess)
      cudaStreamSynchronize(s);
  }
  return v;
}

// The failure path of a bounded wait, on purpose: wait on a barrier that no
// thread ever arrives at, give up after limit_ns, raise the error word.
__global__ void k_selftest_wait(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait_bounded(b, 0, limit_ns) && err) atomicExch(err, 1);
}

int launch_selftest_wait(int64_t limit_ns, void* stream) {
  int* err = device_error_word();
  if (!err) return static_cast<int>(cudaErrorUnknown);
  k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, static_cast<unsigned long long>(limit_ns));
  return static_cast<int>(cudaGetLastError());
}

int launch_kernel(Kind kind, zero_dtype dtype, const LaunchArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((ZERO_DEBUG_BOUNDS || (ZERO_STEP_TMA != 0 && kind == Kind::kStep)) && !a.err) {
    LaunchArgs& w = const_cast<LaunchArgs&>(a);
    w.err = device_error_word();
  }
  if (dtype == ZERO_BF16) return launch_typed<__nv_bfloat16>(kind, a, s);
  return launch_typed<__half>(kind, a, s);
}

}  // namespace zero
