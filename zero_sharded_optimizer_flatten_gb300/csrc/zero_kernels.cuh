// CUDA kernels of the ZeRO sharded optimizer step for sm_103a (GB300).
//
// The step is a streaming element-wise pass: per element it reads N 16-bit
// gradient replicas and the fp32 master/m/v of the owning rank, and writes
// master/m/v and the 16-bit parameter.  It is bound by HBM bandwidth, not by
// arithmetic, so no tensor-core path exists here; what matters is coalesced
// 16-byte accesses, enough bytes in flight per SM, and touching each byte
// once.
//
// Work decomposition: the host cuts each masked rank's owned elements into
// jobs (runs contiguous in both the flat and the shard index space) and the
// jobs into tiles of kTile elements.  A persistent grid (SMs x resident CTAs)
// strides over the tiles; a tile finds its job by binary search in the job
// table held in the kernel's parameter space.  In a vector job each thread
// owns 8 consecutive elements (one 16-byte vector of every 16-bit buffer,
// two of every fp32 buffer); element-wise jobs cover unaligned heads, tails
// and runs whose flat and shard offsets can never be co-aligned.
//
// Arithmetic: the reduction adds the replicas in rank order in binary32 and
// the AdamW update rounds every operation once (__fadd_rn, __fmul_rn,
// __fdiv_rn, __fsqrt_rn: IEEE round-to-nearest, no contraction into FMA),
// so the result does not depend on the launch shape, the bucketing or the
// compiler's scheduling.  16-bit results use the hardware's round-to-nearest
// -even conversions, which keep subnormals.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_internal.h"

namespace zero {

// ---------------------------------------------------------------------------
// 16-bit formats

template <class T>
struct Fmt;

template <>
struct Fmt<__half> {
  static __device__ __forceinline__ void unpack(uint32_t w, float& lo, float& hi) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ float widen(uint16_t x) {
    return __half2float(__ushort_as_half(x));
  }
  static __device__ __forceinline__ uint16_t narrow(float x) {
    return __half_as_ushort(__float2half_rn(x));
  }
};

template <>
struct Fmt<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ float widen(uint16_t x) {
    return __uint_as_float(static_cast<uint32_t>(x) << 16);
  }
  static __device__ __forceinline__ uint16_t narrow(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};

template <class T>
__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  Fmt<T>::unpack(w.x, x[0], x[1]);
  Fmt<T>::unpack(w.y, x[2], x[3]);
  Fmt<T>::unpack(w.z, x[4], x[5]);
  Fmt<T>::unpack(w.w, x[6], x[7]);
}

template <class T>
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(Fmt<T>::pack(x[0], x[1]), Fmt<T>::pack(x[2], x[3]),
                    Fmt<T>::pack(x[4], x[5]), Fmt<T>::pack(x[6], x[7]));
}

// ---------------------------------------------------------------------------
// memory access

// Gradient replicas are read exactly once: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_once16(const void* p) {
  unsigned short r;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ float4 ld_state(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st_state(float* p, const float4& v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

__device__ __forceinline__ void st_vec(void* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// ---------------------------------------------------------------------------
// arithmetic

__device__ __forceinline__ float scale_grad(const LaunchArgs& a, float s) {
  if (a.scale_mode == kScaleMul) return __fmul_rn(s, a.inv_n);
  if (a.scale_mode == kScaleDiv) return __fdiv_rn(s, a.n_f);
  return s;
}

// One AdamW update, every operation rounded once to binary32.
__device__ __forceinline__ void adamw1(const StepScalars& s, float g, float& p, float& m,
                                       float& v) {
  p = __fmul_rn(p, s.d);
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.c1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.c2, __fmul_rn(g, g)));
  const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sb), s.eps);
  p = __fsub_rn(p, __fmul_rn(s.ss, __fdiv_rn(m, den)));
}

// Rank-ordered binary32 sum of the N replicas' 8 elements at flat index f.
// NR > 0: N known at compile time, all N vectors are requested before the
// first add (N outstanding 16-byte loads per thread).  NR == 0: any N.
template <class T, int NR>
__device__ __forceinline__ void reduce8(const LaunchArgs& a, int64_t f, float (&g)[8]) {
  if constexpr (NR > 0) {
    uint4 w[NR];
#pragma unroll
    for (int q = 0; q < NR; ++q)
      w[q] = ld_once(static_cast<const uint16_t*>(a.grads[q]) + f);
    unpack8<T>(w[0], g);
#pragma unroll
    for (int q = 1; q < NR; ++q) {
      float h[8];
      unpack8<T>(w[q], h);
#pragma unroll
      for (int k = 0; k < 8; ++k) g[k] = __fadd_rn(g[k], h[k]);
    }
  } else {
    unpack8<T>(ld_once(static_cast<const uint16_t*>(a.grads[0]) + f), g);
    for (int q = 1; q < a.n_ranks; ++q) {
      float h[8];
      unpack8<T>(ld_once(static_cast<const uint16_t*>(a.grads[q]) + f), h);
#pragma unroll
      for (int k = 0; k < 8; ++k) g[k] = __fadd_rn(g[k], h[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) g[k] = scale_grad(a, g[k]);
}

template <class T, int NR>
__device__ __forceinline__ float reduce1(const LaunchArgs& a, int64_t f) {
  const int n = NR > 0 ? NR : a.n_ranks;
  float g = Fmt<T>::widen(ld_once16(static_cast<const uint16_t*>(a.grads[0]) + f));
#pragma unroll
  for (int q = 1; q < n; ++q)
    g = __fadd_rn(g, Fmt<T>::widen(ld_once16(static_cast<const uint16_t*>(a.grads[q]) + f)));
  return scale_grad(a, g);
}

// ---------------------------------------------------------------------------
// tile -> job

__device__ __forceinline__ int find_job(const LaunchArgs& a, int64_t tile) {
  int lo = 0, hi = a.n_jobs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.jobs[mid].tile_begin <= tile)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Calls body_vec(job, e) for the 8-element vector at job offset e, or
// body_one(job, e) for single elements, over every tile of the launch.
template <class BodyVec, class BodyOne>
__device__ __forceinline__ void for_each_tile(const LaunchArgs& a, BodyVec body_vec,
                                              BodyOne body_one) {
  for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
    const Job& jb = a.jobs[find_job(a, tile)];
    const int64_t base = (tile - jb.tile_begin) * kTile;
    if (jb.vec) {
      const int64_t e = base + static_cast<int64_t>(threadIdx.x) * kVec;
      if (e < jb.len) body_vec(jb, e);
    } else {
#pragma unroll 1
      for (int k = 0; k < kVec; ++k) {
        const int64_t e = base + k * kThreads + threadIdx.x;
        if (e < jb.len) body_one(jb, e);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// kernels

// Fused step: reduce-scatter + AdamW + cast + all-gather.
template <class T, int NR>
__global__ void __launch_bounds__(kThreads) k_step(const __grid_constant__ LaunchArgs a) {
  for_each_tile(
      a,
      [&](const Job& jb, int64_t e) {
        const int64_t f = jb.flat_off + e, i = jb.shard_off + e;
        const int r = jb.rank;
        float* pm = a.master[r] + i;
        float* mm = a.m[r] + i;
        float* vm = a.v[r] + i;
        float g[8];
        reduce8<T, NR>(a, f, g);
        const float4 p0 = ld_state(pm), p1 = ld_state(pm + 4);
        const float4 m0 = ld_state(mm), m1 = ld_state(mm + 4);
        const float4 v0 = ld_state(vm), v1 = ld_state(vm + 4);
        float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) adamw1(a.sc, g[k], p[k], m[k], v[k]);
        st_state(pm, make_float4(p[0], p[1], p[2], p[3]));
        st_state(pm + 4, make_float4(p[4], p[5], p[6], p[7]));
        st_state(mm, make_float4(m[0], m[1], m[2], m[3]));
        st_state(mm + 4, make_float4(m[4], m[5], m[6], m[7]));
        st_state(vm, make_float4(v[0], v[1], v[2], v[3]));
        st_state(vm + 4, make_float4(v[4], v[5], v[6], v[7]));
        const uint4 o = pack8<T>(p);
        if (a.full16) st_vec(static_cast<uint16_t*>(a.full16) + f, o);
        if (a.shard16[r]) st_vec(static_cast<uint16_t*>(a.shard16[r]) + i, o);
      },
      [&](const Job& jb, int64_t e) {
        const int64_t f = jb.flat_off + e, i = jb.shard_off + e;
        const int r = jb.rank;
        const float g = reduce1<T, NR>(a, f);
        float p = a.master[r][i], m = a.m[r][i], v = a.v[r][i];
        adamw1(a.sc, g, p, m, v);
        a.master[r][i] = p;
        a.m[r][i] = m;
        a.v[r][i] = v;
        const uint16_t o = Fmt<T>::narrow(p);
        if (a.full16) static_cast<uint16_t*>(a.full16)[f] = o;
        if (a.shard16[r]) static_cast<uint16_t*>(a.shard16[r])[i] = o;
      });
}

// Reduce-scatter alone: fp32 gradient shards.
template <class T, int NR>
__global__ void __launch_bounds__(kThreads) k_reduce_scatter(const __grid_constant__ LaunchArgs a) {
  for_each_tile(
      a,
      [&](const Job& jb, int64_t e) {
        float g[8];
        reduce8<T, NR>(a, jb.flat_off + e, g);
        float* out = a.gshard[jb.rank] + jb.shard_off + e;
        st_state(out, make_float4(g[0], g[1], g[2], g[3]));
        st_state(out + 4, make_float4(g[4], g[5], g[6], g[7]));
      },
      [&](const Job& jb, int64_t e) {
        a.gshard[jb.rank][jb.shard_off + e] = reduce1<T, NR>(a, jb.flat_off + e);
      });
}

// AdamW + cast on fp32 gradient shards.
template <class T>
__global__ void __launch_bounds__(kThreads) k_adamw(const __grid_constant__ LaunchArgs a) {
  for_each_tile(
      a,
      [&](const Job& jb, int64_t e) {
        const int64_t i = jb.shard_off + e;
        const int r = jb.rank;
        float* pm = a.master[r] + i;
        float* mm = a.m[r] + i;
        float* vm = a.v[r] + i;
        const float* gm = a.gshard[r] + i;
        const float4 g0 = ld_state(gm), g1 = ld_state(gm + 4);
        const float4 p0 = ld_state(pm), p1 = ld_state(pm + 4);
        const float4 m0 = ld_state(mm), m1 = ld_state(mm + 4);
        const float4 v0 = ld_state(vm), v1 = ld_state(vm + 4);
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) adamw1(a.sc, g[k], p[k], m[k], v[k]);
        st_state(pm, make_float4(p[0], p[1], p[2], p[3]));
        st_state(pm + 4, make_float4(p[4], p[5], p[6], p[7]));
        st_state(mm, make_float4(m[0], m[1], m[2], m[3]));
        st_state(mm + 4, make_float4(m[4], m[5], m[6], m[7]));
        st_state(vm, make_float4(v[0], v[1], v[2], v[3]));
        st_state(vm + 4, make_float4(v[4], v[5], v[6], v[7]));
        if (a.shard16[r]) st_vec(static_cast<uint16_t*>(a.shard16[r]) + i, pack8<T>(p));
      },
      [&](const Job& jb, int64_t e) {
        const int64_t i = jb.shard_off + e;
        const int r = jb.rank;
        float p = a.master[r][i], m = a.m[r][i], v = a.v[r][i];
        adamw1(a.sc, a.gshard[r][i], p, m, v);
        a.master[r][i] = p;
        a.m[r][i] = m;
        a.v[r][i] = v;
        if (a.shard16[r]) static_cast<uint16_t*>(a.shard16[r])[i] = Fmt<T>::narrow(p);
      });
}

// All-gather: copy each rank's 16-bit shard into the flat buffer.
template <class T>
__global__ void __launch_bounds__(kThreads) k_allgather(const __grid_constant__ LaunchArgs a) {
  for_each_tile(
      a,
      [&](const Job& jb, int64_t e) {
        const uint4 w = ld_once(static_cast<const uint16_t*>(a.shard16[jb.rank]) + jb.shard_off + e);
        st_vec(static_cast<uint16_t*>(a.full16) + jb.flat_off + e, w);
      },
      [&](const Job& jb, int64_t e) {
        static_cast<uint16_t*>(a.full16)[jb.flat_off + e] =
            ld_once16(static_cast<const uint16_t*>(a.shard16[jb.rank]) + jb.shard_off + e);
      });
}

// Initialise a rank's fp32 master from its 16-bit partition; zero m and v.
template <class T>
__global__ void __launch_bounds__(kThreads) k_init(const __grid_constant__ LaunchArgs a) {
  for_each_tile(
      a,
      [&](const Job& jb, int64_t e) {
        const int64_t i = jb.shard_off + e;
        const int r = jb.rank;
        float p[8];
        unpack8<T>(ld_once(static_cast<const uint16_t*>(a.full16) + jb.flat_off + e), p);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        st_state(a.master[r] + i, make_float4(p[0], p[1], p[2], p[3]));
        st_state(a.master[r] + i + 4, make_float4(p[4], p[5], p[6], p[7]));
        st_state(a.m[r] + i, z);
        st_state(a.m[r] + i + 4, z);
        st_state(a.v[r] + i, z);
        st_state(a.v[r] + i + 4, z);
      },
      [&](const Job& jb, int64_t e) {
        const int64_t i = jb.shard_off + e;
        const int r = jb.rank;
        a.master[r][i] =
            Fmt<T>::widen(ld_once16(static_cast<const uint16_t*>(a.full16) + jb.flat_off + e));
        a.m[r][i] = 0.f;
        a.v[r][i] = 0.f;
      });
}

// ---------------------------------------------------------------------------
// launch (host)

// Grid of a persistent launch of kernel `fn`: resident CTAs per SM times the
// SM count of the current device, capped by the tile count.
int persistent_grid(const void* fn, int64_t n_tiles);

template <class T, template <class, int> class Pick>
const void* by_ranks(int n) {
  switch (n) {
    case 1: return Pick<T, 1>::get();
    case 2: return Pick<T, 2>::get();
    case 3: return Pick<T, 3>::get();
    case 4: return Pick<T, 4>::get();
    case 5: return Pick<T, 5>::get();
    case 6: return Pick<T, 6>::get();
    case 7: return Pick<T, 7>::get();
    case 8: return Pick<T, 8>::get();
    default: return Pick<T, 0>::get();
  }
}

template <class T, int NR>
struct PickStep {
  static const void* get() { return reinterpret_cast<const void*>(&k_step<T, NR>); }
};

template <class T, int NR>
struct PickReduce {
  static const void* get() { return reinterpret_cast<const void*>(&k_reduce_scatter<T, NR>); }
};

template <class T>
int launch_typed(Kind kind, const LaunchArgs& a, cudaStream_t s) {
  const void* fn = nullptr;
  switch (kind) {
    case Kind::kStep: fn = by_ranks<T, PickStep>(a.n_ranks); break;
    case Kind::kReduceScatter: fn = by_ranks<T, PickReduce>(a.n_ranks); break;
    case Kind::kAdamw: fn = reinterpret_cast<const void*>(&k_adamw<T>); break;
    case Kind::kAllgather: fn = reinterpret_cast<const void*>(&k_allgather<T>); break;
    case Kind::kInit: fn = reinterpret_cast<const void*>(&k_init<T>); break;
  }
  const int grid = persistent_grid(fn, a.n_tiles);
  if (grid <= 0) return static_cast<int>(cudaGetLastError());
  void* args[] = {const_cast<LaunchArgs*>(&a)};
  return static_cast<int>(cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, 0, s));
}

}  // namespace zero
