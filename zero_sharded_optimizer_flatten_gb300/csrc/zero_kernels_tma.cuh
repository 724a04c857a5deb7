// The fused step with bulk-copy (TMA) staging, for sm_103a.
//
// A persistent CTA walks the tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// One elected thread moves each tile's inputs -- the N 16-bit gradient
// slices and the fp32 master/m/v slices, each one contiguous run -- from
// global into a ring of shared-memory stages with 1-D cp.async.bulk copies
// that complete on the stage's mbarrier (transaction bytes); the ring keeps
// kTmaStages tiles in flight, so the loads of later tiles overlap the
// arithmetic and the stores of the current one.  The consumers read the
// stage in the same two-quad layout as the plain kernel and store results
// straight to global memory.
//
// Every wait is bounded: thread 0 polls the mbarrier for at most one second
// (%globaltimer); if it gives up it raises the device error word (read by
// zero_sync as ZERO_ERR_TIMEOUT), waits a bounded time for the copies it
// issued, and the CTA returns.  The other threads only wait at CTA barriers.
#pragma once

#include "zero_kernels.cuh"

#ifndef ZERO_TMA_STAGES
#define ZERO_TMA_STAGES 2
#endif

namespace zero {

constexpr int kTmaStages = ZERO_TMA_STAGES;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // one second

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
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :
      : "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint2 lds8(uint32_t a) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
  return r;
}

__device__ __forceinline__ float4 lds16f(uint32_t a) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(a));
  return r;
}

// Shared-memory bytes of one stage for NR replicas.
template <int NR>
constexpr int tma_stage_bytes() {
  return kTile * (2 * NR + 12);
}

template <class T, int NR>
__global__ void __launch_bounds__(kThreads, 1) k_step_tma(const __grid_constant__ LaunchArgs a) {
  grid_dependency_begin();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) unsigned long long full_bar[kTmaStages];
  __shared__ int ok;
  constexpr int kStage = tma_stage_bytes<NR>();
  const uint32_t base_addr = smem_addr(smem);
  const int64_t my_n = (a.n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full_bar[s])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ok = 1;
  }
  __syncthreads();

  // thread 0: bring tile k of this CTA into stage k % kTmaStages
  auto issue = [&](int64_t k) {
    const int64_t tile = blockIdx.x + k * gridDim.x;
    const Job& jb = a.jobs[find_job(a, tile)];
    const int64_t base = (tile - jb.tile_begin) * kTile;
    const int64_t cnt = jb.len - base < kTile ? jb.len - base : kTile;
    const int s = static_cast<int>(k % kTmaStages);
    const uint32_t bar = smem_addr(&full_bar[s]);
    const uint32_t dst = base_addr + s * kStage;
    const uint32_t bytes = static_cast<uint32_t>(cnt * (2 * NR + 12));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    const int64_t f = jb.flat_off + base, i = jb.shard_off + base;
    if (!access_ok(a, jb, base, cnt)) return;  // bounds-checked builds only
#pragma unroll
    for (int q = 0; q < NR; ++q)
      bulk_g2s(dst + q * kTile * 2, static_cast<const uint16_t*>(a.grads[q]) + f,
               static_cast<uint32_t>(cnt * 2), bar);
    const uint32_t st = dst + NR * kTile * 2;
    bulk_g2s(st, a.master[jb.rank] + i, static_cast<uint32_t>(cnt * 4), bar);
    bulk_g2s(st + kTile * 4, a.m[jb.rank] + i, static_cast<uint32_t>(cnt * 4), bar);
    bulk_g2s(st + 2 * kTile * 4, a.v[jb.rank] + i, static_cast<uint32_t>(cnt * 4), bar);
  };

  if (threadIdx.x == 0)
    for (int64_t k = 0; k < my_n && k < kTmaStages; ++k) issue(k);

  int64_t issued = my_n < kTmaStages ? my_n : kTmaStages;
  int64_t k_fail = -1;
  for (int64_t k = 0; k < my_n; ++k) {
    const int s = static_cast<int>(k % kTmaStages);
    const uint32_t parity = static_cast<uint32_t>((k / kTmaStages) & 1);
    const uint32_t bar = smem_addr(&full_bar[s]);
    if (threadIdx.x == 0 && !mbar_wait_bounded(bar, parity)) {
      ok = 0;
      if (a.err) atomicExch(a.err, 1);
    }
    __syncthreads();
    if (!ok) {
      k_fail = k;
      break;
    }
    // thread 0 saw this phase complete, so this returns at the first poll; every
    // thread still observes the barrier itself before it reads the stage
    if (!mbar_wait_bounded(bar, parity) && a.err) atomicExch(a.err, 1);

    const int64_t tile = blockIdx.x + k * gridDim.x;
    const Job& jb = a.jobs[find_job(a, tile)];
    const int64_t base = (tile - jb.tile_begin) * kTile;
    const int64_t cnt = jb.len - base < kTile ? jb.len - base : kTile;
    const int e0 = threadIdx.x * kVec;
    if (e0 < cnt) {
      const bool two = e0 + kHalf < cnt;
      const int r = jb.rank;
      const uint32_t dst = base_addr + s * kStage;
      float g[8], p[8], m[8], v[8];
      {
        const uint2 z = make_uint2(0u, 0u);
        uint2 w0[NR], w1[NR];
#pragma unroll
        for (int q = 0; q < NR; ++q) {
          w0[q] = lds8(dst + q * kTile * 2 + e0 * 2);
          w1[q] = two ? lds8(dst + q * kTile * 2 + (e0 + kHalf) * 2) : z;
        }
        unpack4<T>(w0[0], g);
        unpack4<T>(w1[0], g + 4);
#pragma unroll
        for (int q = 1; q < NR; ++q) {
          float h[8];
          unpack4<T>(w0[q], h);
          unpack4<T>(w1[q], h + 4);
#pragma unroll
          for (int j = 0; j < 8; ++j) g[j] = __fadd_rn(g[j], h[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = scale_grad(a, g[j]);
      }
      const uint32_t st = dst + NR * kTile * 2;
      const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
      split(lds16f(st + e0 * 4), p);
      split(two ? lds16f(st + (e0 + kHalf) * 4) : zf, p + 4);
      split(lds16f(st + kTile * 4 + e0 * 4), m);
      split(two ? lds16f(st + kTile * 4 + (e0 + kHalf) * 4) : zf, m + 4);
      split(lds16f(st + 2 * kTile * 4 + e0 * 4), v);
      split(two ? lds16f(st + 2 * kTile * 4 + (e0 + kHalf) * 4) : zf, v + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) adamw1(a.sc, g[j], p[j], m[j], v[j]);
      const int64_t f0 = jb.flat_off + base + e0, i0 = jb.shard_off + base + e0;
      store_state2(a.master[r], i0, i0 + kHalf, two, p);
      store_state2(a.m[r], i0, i0 + kHalf, two, m);
      store_state2(a.v[r], i0, i0 + kHalf, two, v);
      if (a.full16) store_16x2<T>(a.full16, f0, f0 + kHalf, two, p);
      if (a.shard16[r]) store_16x2<T>(a.shard16[r], i0, i0 + kHalf, two, p);
    }
    __syncthreads();  // stage s is free again
    if (threadIdx.x == 0 && issued < my_n) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(issued);
      ++issued;
    }
  }
  if (k_fail >= 0 && threadIdx.x == 0) {
    // give the copies still in flight (tiles k_fail .. issued-1) a bounded
    // time to land before the CTA and its shared memory go away
    for (int64_t k = k_fail; k < issued; ++k) {
      const uint32_t bar = smem_addr(&full_bar[k % kTmaStages]);
      if (!mbar_wait_bounded(bar, static_cast<uint32_t>((k / kTmaStages) & 1))) break;
    }
  }
}

template <class T, int NR>
struct PickStepTma {
  static const void* get() { return reinterpret_cast<const void*>(&k_step_tma<T, NR>); }
};

// Persistent grid: resident CTAs per SM (given the stage ring's shared
// memory) times the SM count, capped by the tile count.
int resident_grid(const void* fn, int smem_bytes, int64_t n_tiles);

template <class T>
int launch_step_tma_impl(const LaunchArgs& a, cudaStream_t s) {
  const void* fn = nullptr;
  int smem = 0;
  switch (a.n_ranks) {
    case 1: fn = PickStepTma<T, 1>::get(); smem = tma_stage_bytes<1>(); break;
    case 2: fn = PickStepTma<T, 2>::get(); smem = tma_stage_bytes<2>(); break;
    case 3: fn = PickStepTma<T, 3>::get(); smem = tma_stage_bytes<3>(); break;
    case 4: fn = PickStepTma<T, 4>::get(); smem = tma_stage_bytes<4>(); break;
    case 5: fn = PickStepTma<T, 5>::get(); smem = tma_stage_bytes<5>(); break;
    case 6: fn = PickStepTma<T, 6>::get(); smem = tma_stage_bytes<6>(); break;
    case 7: fn = PickStepTma<T, 7>::get(); smem = tma_stage_bytes<7>(); break;
    default: fn = PickStepTma<T, 8>::get(); smem = tma_stage_bytes<8>(); break;
  }
  smem *= kTmaStages;
  const int grid = resident_grid(fn, smem, a.n_tiles);
  if (grid <= 0) return static_cast<int>(cudaGetLastError());
  void* args[] = {const_cast<LaunchArgs*>(&a)};
  return static_cast<int>(launch_ordered(fn, dim3(grid), dim3(kThreads), args,
                                           static_cast<size_t>(smem), s));
}

}  // namespace zero
