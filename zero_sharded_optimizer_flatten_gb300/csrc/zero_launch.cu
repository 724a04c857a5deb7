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

// The decision of the mixed-precision step: sum the per-tile partials in a
// fixed order (binary32 pairs, see SqSum), then update the loss-scale state
// and form the step's coefficient and AdamW constants (binary64, each
// rounded once).  beta1^t and beta2^t come from the reduction kernel.
constexpr int kFinUnroll = 8;  // partial loads in flight per thread

__device__ void amp_decide(zero_amp_state& x, double sumsq, const AmpParams& p, double b1t,
                           double b2t) {
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
  const zero_adamw_hparams& h = p.hp;
  x.sc[0] = static_cast<float>(1.0 - h.lr * h.weight_decay);
  x.sc[1] = static_cast<float>(h.beta1);
  x.sc[2] = static_cast<float>(h.beta2);
  x.sc[3] = static_cast<float>(1.0 - h.beta1);
  x.sc[4] = static_cast<float>(1.0 - h.beta2);
  x.sc[5] = static_cast<float>(h.lr / (1.0 - b1t));
  x.sc[6] = static_cast<float>(sqrt(1.0 - b2t));
  x.sc[7] = static_cast<float>(h.eps);
  x.overflow = 0;
  x.step = x.step + 1;
  x.good_steps += 1;
  if (p.cfg.window > 0 && x.good_steps >= p.cfg.window) {
    x.scale = S * 2.0;
    x.good_steps = 0;
    x.hysteresis_left = p.cfg.hysteresis;
  }
}

// kFinCtas CTAs: CTA c's thread t adds partials j = c*T + t, j + C*T, ... in
// increasing order; the CTA adds its threads (shuffle trees, then the warps
// in index order) and publishes its sum; the CTA that arrives last (atomic
// counter, no waiting) adds the CTAs' sums in index order and decides.
__global__ void __launch_bounds__(kFinThreads) k_amp_finalize(const NormPartial* partials,
                                                              int64_t n, zero_amp_state* st,
                                                              AmpHead* head, const AmpParams p) {
  constexpr int64_t kAll = static_cast<int64_t>(kFinCtas) * kFinThreads;
  const float4* src = reinterpret_cast<const float4*>(partials);
  SqSum s = sq_zero();
  // kFinUnroll of the thread's partials in flight at once (the last group
  // predicated), added in increasing index order
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x; i < n;
       i += kFinUnroll * kAll) {
    float4 q[kFinUnroll];
#pragma unroll
    for (int k = 0; k < kFinUnroll; ++k)
      q[k] = i + k * kAll < n ? __ldcg(src + i + k * kAll) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kFinUnroll; ++k)
      if (i + k * kAll < n) s.add(q[k]);
  }
  __shared__ SqSum warp_part[kFinThreads / 32];
  __shared__ int last;
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    SqSum t = warp_part[0];
    for (int w = 1; w < kFinThreads / 32; ++w) t.add(warp_part[w]);
    store_partial(&head->cta_part[blockIdx.x], t);
    __threadfence();
    last = atomicAdd(&head->arrived, 1) == kFinCtas - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  __shared__ AmpBcast rec;
  if (threadIdx.x < 32) {
    SqSum c = sq_zero();
    if (threadIdx.x < kFinCtas) c.add(__ldcg(reinterpret_cast<const float4*>(head->cta_part) + threadIdx.x));
    c = warp_sum(c);
    if (threadIdx.x == 0) {
      zero_amp_state x = *st;
      amp_decide(x, c.value(), p, __ldcg(&head->beta_pow[0]), __ldcg(&head->beta_pow[1]));
      *st = x;
      head->arrived = 0;
      AmpBcast b = {};
      b.overflow = x.overflow;
      b.coef = x.coef;
      for (int k = 0; k < 8; ++k) b.sc[k] = x.sc[k];
      rec = b;
    }
  }
  __syncthreads();
  // the decision record to its kAmpCopies places, one thread each
  if (threadIdx.x < kAmpCopies) head->bcast[threadIdx.x] = rec;
}

__global__ void k_amp_init(zero_amp_state* st, const zero_amp_state v) { *st = v; }

int launch_amp_finalize(const NormPartial* partials, int64_t n_tiles, zero_amp_state* state,
                        AmpHead* head, const AmpParams& p, void* stream) {
  AmpParams params = p;
  void* args[] = {const_cast<NormPartial**>(&partials), &n_tiles, &state, &head, &params};
  return static_cast<int>(cudaLaunchKernel(reinterpret_cast<const void*>(&k_amp_finalize),
                                           dim3(kFinCtas), dim3(kFinThreads), args, 0,
                                           static_cast<cudaStream_t>(stream)));
}

int launch_amp_init(zero_amp_state* state, const zero_amp_state& init, void* stream) {
  k_amp_init<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(state, init);
  return static_cast<int>(cudaGetLastError());
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

// Bounded waits on a shared-memory mbarrier (the self-test below).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Poll the barrier's phase `parity` for at most limit_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
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
  if (ZERO_DEBUG_BOUNDS && !a.err) {
    LaunchArgs& w = const_cast<LaunchArgs&>(a);
    w.err = device_error_word();
  }
  if (dtype == ZERO_BF16) return launch_typed<__nv_bfloat16>(kind, a, s);
  return launch_typed<__half>(kind, a, s);
}

}  // namespace zero
