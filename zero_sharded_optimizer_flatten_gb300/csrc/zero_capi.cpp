// C-ABI device calls of the ZeRO sharded optimizer step: argument checks,
// the per-step AdamW constants, the job tables and the launches.
//
// What each call computes is documented in include/zero.h; the sources are
// "DeepSpeed ZeRO-2 ... DeepSpeedZeroOptimizer" (discosf.com) §4.1-§4.4 for
// init / reduce-scatter / local update / all-gather, and "ZeRO 优化器"
// (cookllm.com) 梯度同步 for the summed (rather than averaged) reduction.
#include <cuda_runtime.h>
#include <inttypes.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "zero_capi_util.h"
#include "zero_host.h"
#include "zero_internal.h"

namespace zero {

constexpr int kMaxHostThreads = 1024;    // host threads of one host optimizer call
constexpr int kMaxOffloadChunks = 4096;  // chunks (one event each) of one offload step

char* error_buffer() {
  static thread_local char buf[1024];
  return buf;
}

std::atomic<int64_t> g_launches{0};

// The binary32 constants of step t, each formed in binary64 and rounded once.
StepScalars make_scalars(const zero_adamw_hparams& h, int64_t t) {
  StepScalars s;
  s.d = static_cast<float>(1.0 - h.lr * h.weight_decay);
  s.b1 = static_cast<float>(h.beta1);
  s.b2 = static_cast<float>(h.beta2);
  s.c1 = static_cast<float>(1.0 - h.beta1);
  s.c2 = static_cast<float>(1.0 - h.beta2);
  s.ss = static_cast<float>(h.lr / (1.0 - pow(h.beta1, static_cast<double>(t))));
  s.sb = static_cast<float>(sqrt(1.0 - pow(h.beta2, static_cast<double>(t))));
  s.eps = static_cast<float>(h.eps);
  return s;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

zero_status check_plan_mask(const char* fn, const zero_plan* plan, uint64_t rank_mask) {
  if (!plan) return fail(ZERO_ERR_INVALID, "%s: plan is NULL", fn);
  if (rank_mask == 0) return fail(ZERO_ERR_INVALID, "%s: rank_mask selects no rank", fn);
  if (plan->n_ranks < 64 && (rank_mask >> plan->n_ranks) != 0)
    return fail(ZERO_ERR_INVALID, "%s: rank_mask 0x%" PRIx64 " names a rank >= n_ranks (%d)", fn,
                rank_mask, plan->n_ranks);
  return ZERO_OK;
}

bool in_mask(uint64_t mask, int r) { return (mask >> r) & 1u; }

zero_status check_dtype(const char* fn, zero_dtype dtype) {
  if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return fail(ZERO_ERR_INVALID, "%s: unknown dtype", fn);
  return ZERO_OK;
}

// Per-rank pointer array: every masked rank's entry non-NULL (unless
// nullable) and 16-byte aligned.  all_ranks: the entries are the flat
// gradient replicas, which every rank must supply unless the flat buffer is
// empty.
template <class P>
zero_status check_ptrs(const char* fn, const char* what, P const* arr, const zero_plan* plan,
                       uint64_t mask, bool nullable_entries, bool all_ranks = false) {
  if (!arr) return fail(ZERO_ERR_INVALID, "%s: %s is NULL", fn, what);
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!all_ranks && !in_mask(mask, r)) continue;
    if (!all_ranks && plan->shard_len[r] == 0) continue;  // an empty shard is never touched
    if (all_ranks && plan->padded == 0) continue;          // nor is an empty flat buffer
    const void* p = arr[r];
    if (!p) {
      if (nullable_entries) continue;
      return fail(ZERO_ERR_INVALID, "%s: %s[%d] is NULL", fn, what, r);
    }
    if (!aligned16(p)) return fail(ZERO_ERR_ALIGN, "%s: %s[%d] is not 16-byte aligned", fn, what, r);
  }
  return ZERO_OK;
}

zero_status check_hparams(const char* fn, const zero_adamw_hparams* hp, int64_t step) {
  if (!hp) return fail(ZERO_ERR_INVALID, "%s: hparams is NULL", fn);
  const double vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  for (double x : vals)
    if (!isfinite(x)) return fail(ZERO_ERR_INVALID, "%s: non-finite hyper-parameter", fn);
  if (hp->lr < 0 || hp->weight_decay < 0 || !(hp->eps > 0))
    return fail(ZERO_ERR_INVALID, "%s: need lr >= 0, weight_decay >= 0, eps > 0", fn);
  if (hp->beta1 < 0 || hp->beta1 >= 1 || hp->beta2 < 0 || hp->beta2 >= 1)
    return fail(ZERO_ERR_INVALID, "%s: betas must lie in [0, 1)", fn);
  if (step < 1) return fail(ZERO_ERR_INVALID, "%s: step must be >= 1 (got %" PRId64 ")", fn, step);
  return ZERO_OK;
}

void set_scale(LaunchArgs& a, int n_ranks, zero_reduce_op op) {
  a.n_ranks = n_ranks;
  a.n_f = static_cast<float>(n_ranks);
  a.inv_n = 1.0f / static_cast<float>(n_ranks);
  if (op == ZERO_REDUCE_SUM || n_ranks == 1)
    a.scale_mode = kScaleNone;
  else if ((n_ranks & (n_ranks - 1)) == 0)
    a.scale_mode = kScaleMul;  // 1/N exact
  else
    a.scale_mode = kScaleDiv;
}

// Split one run into vector and element-wise jobs.
void add_run(std::vector<Job>& out, int r, int64_t flat, int64_t shard, int64_t len) {
  if (len <= 0) return;
  if ((flat - shard) % kVec != 0) {  // flat and shard never co-aligned
    out.push_back({flat, shard, len, 0, r, 0});
    return;
  }
  int64_t head = (kVec - flat % kVec) % kVec;
  if (head > len) head = len;
  if (head) out.push_back({flat, shard, head, 0, r, 0});
  const int64_t body = (len - head) / kVec * kVec;
  if (body) out.push_back({flat + head, shard + head, body, 0, r, 1});
  const int64_t tail = len - head - body;
  if (tail) out.push_back({flat + head + body, shard + head + body, tail, 0, r, 0});
}

// Jobs of the masked ranks restricted to the flat range [lo, hi).
void build_jobs(const zero_plan* plan, uint64_t mask, int64_t lo, int64_t hi,
                std::vector<Job>& jobs) {
  jobs.clear();
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!in_mask(mask, r)) continue;
    for (const auto& run : plan->runs[r]) {
      const int64_t a = std::max(lo, run.flat_off);
      const int64_t b = std::min(hi, run.flat_off + run.len);
      if (a < b) add_run(jobs, r, a, run.shard_off + (a - run.flat_off), b - a);
    }
  }
}

// Launch `kind` over `jobs`, at most kMaxJobs per launch.  `tiles_done`
// (nullable) numbers the tiles across launches: each launch's first tile is
// given index *tiles_done (LaunchArgs::tile_base), which then advances.
// The first launch is ordered after everything before it on the stream when
// a.early is 0 on entry; every later one is launched early (its jobs are
// disjoint from the ones before it; see grid_dependency_begin).
zero_status launch_jobs(const char* fn, Kind kind, zero_dtype dtype, LaunchArgs& a,
                        const std::vector<Job>& jobs, void* stream, int64_t* tiles_done) {
  size_t j0 = 0;
  while (j0 < jobs.size()) {
    const size_t nj = std::min<size_t>(jobs.size() - j0, kMaxJobs);
    int64_t tiles = 0;
    for (size_t j = 0; j < nj; ++j) {
      a.jobs[j] = jobs[j0 + j];
      a.jobs[j].tile_begin = tiles;
      tiles += (a.jobs[j].len + kTile - 1) / kTile;
    }
    a.n_jobs = static_cast<int32_t>(nj);
    a.n_tiles = tiles;
    a.tile_base = tiles_done ? *tiles_done : 0;
    const int err = launch_kernel(kind, dtype, a, stream);
    if (err != 0)
      return fail(ZERO_ERR_CUDA, "%s: launch failed: %s", fn,
                  cudaGetErrorString(static_cast<cudaError_t>(err)));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    a.early = 1;  // the next launch of this run touches other elements
    if (tiles_done) *tiles_done += tiles;
    j0 += nj;
  }
  return ZERO_OK;
}

// The buffer lengths the bounds-checked build verifies every access against.
void set_bounds(LaunchArgs& a, const zero_plan* plan) {
  a.flat_len = plan->padded;
  for (int r = 0; r < plan->n_ranks; ++r) a.shard_len[r] = plan->shard_len[r];
}

// Run `kind` bucket by bucket over the flat index space.
zero_status run_buckets(const char* fn, Kind kind, zero_dtype dtype, const zero_plan* plan,
                        uint64_t mask, int64_t bucket, LaunchArgs& a, void* stream,
                        int64_t* tiles_done = nullptr) {
  set_bounds(a, plan);
  a.early = 0;  // the run's first launch waits for all earlier work on the stream
  std::vector<Job> jobs;
  const int64_t total = plan->padded;
  const int64_t B = bucket > 0 ? bucket : std::max<int64_t>(total, 1);
  // Only buckets that meet a masked rank's run launch anything.
  for (int64_t lo = 0; lo < total; lo += B) {
    const int64_t hi = std::min(total, lo + B);
    build_jobs(plan, mask, lo, hi, jobs);
    if (jobs.empty()) continue;
    const zero_status st = launch_jobs(fn, kind, dtype, a, jobs, stream, tiles_done);
    if (st != ZERO_OK) return st;
  }
  return ZERO_OK;
}

// Tiles run_buckets would launch for this mask and bucketing.
int64_t count_tiles(const zero_plan* plan, uint64_t mask, int64_t bucket) {
  std::vector<Job> jobs;
  const int64_t total = plan->padded;
  const int64_t B = bucket > 0 ? bucket : std::max<int64_t>(total, 1);
  int64_t tiles = 0;
  for (int64_t lo = 0; lo < total; lo += B) {
    build_jobs(plan, mask, lo, std::min(total, lo + B), jobs);
    for (const Job& j : jobs) tiles += (j.len + kTile - 1) / kTile;
  }
  return tiles;
}

zero_status check_amp_config(const char* fn, const zero_amp_config* c) {
  if (!c) return fail(ZERO_ERR_INVALID, "%s: cfg is NULL", fn);
  if (!isfinite(c->init_scale) || !(c->init_scale > 0) || !isfinite(c->min_scale) ||
      !(c->min_scale > 0))
    return fail(ZERO_ERR_INVALID, "%s: init_scale and min_scale must be finite and > 0", fn);
  if (c->window < 0 || c->hysteresis < 1)
    return fail(ZERO_ERR_INVALID, "%s: need window >= 0 and hysteresis >= 1", fn);
  if (!isfinite(c->max_norm)) return fail(ZERO_ERR_INVALID, "%s: max_norm must be finite", fn);
  return ZERO_OK;
}

zero_status pending_error(const char* fn) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(ZERO_ERR_CUDA, "%s: pending CUDA error: %s", fn, cudaGetErrorString(e));
  return ZERO_OK;
}

LaunchArgs* new_args() {
  LaunchArgs* a = new (std::nothrow) LaunchArgs;
  if (a) memset(a, 0, sizeof(LaunchArgs));
  return a;
}

// One host update piece: elements [off, off + len) of rank r's shard.
struct HostPiece {
  int r;
  int64_t off, len;
};

// The host optimizer's operands (host arrays, per rank).
struct HostUpdate {
  StepScalars sc;
  zero_dtype dtype;
  float* const* master;
  float* const* m;
  float* const* v;
  const float* const* grad_shards;
  void* const* out16;   // nullable; entries nullable
  bool scaled = false;  // mixed precision: the gradient is multiplied by coef first
  float coef = 1.0f;

  // Update elements [b0, b1) of the concatenation of `pieces`.
  void slice(const std::vector<HostPiece>& pieces, int64_t b0, int64_t b1) const {
    int64_t seen = 0;
    for (const HostPiece& pc : pieces) {
      if (seen >= b1) break;
      const int64_t lo = std::max(b0, seen), hi = std::min(b1, seen + pc.len);
      if (lo < hi) {
        const int64_t o = pc.off + (lo - seen);
        uint16_t* o16 = out16 && out16[pc.r] ? static_cast<uint16_t*>(out16[pc.r]) + o : nullptr;
        if (scaled)
          cpu_adamw_range_scaled(sc, coef, dtype, master[pc.r] + o, m[pc.r] + o, v[pc.r] + o,
                                 grad_shards[pc.r] + o, o16, hi - lo);
        else
          cpu_adamw_range(sc, dtype, master[pc.r] + o, m[pc.r] + o, v[pc.r] + o,
                          grad_shards[pc.r] + o, o16, hi - lo);
      }
      seen += pc.len;
    }
  }
};

struct ArgsHolder {
  LaunchArgs* p;
  explicit ArgsHolder(LaunchArgs* q) : p(q) {}
  ~ArgsHolder() { delete p; }
};

}  // namespace
}  // namespace zero

using namespace zero;

#define ZERO_TRY(x)                    \
  do {                                 \
    const zero_status st_ = (x);       \
    if (st_ != ZERO_OK) return st_;    \
  } while (0)

extern "C" zero_status zero_init_shards(const zero_plan* plan, const void* full_flat16,
                                        zero_dtype dtype, float* const* master, float* const* m,
                                        float* const* v, uint64_t rank_mask, void* stream) {
  const char* fn = "zero_init_shards";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (!full_flat16 && plan->padded > 0)
    return fail(ZERO_ERR_INVALID, "%s: full_flat16 is NULL", fn);
  if (!aligned16(full_flat16)) return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!in_mask(rank_mask, r)) continue;
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
  }
  a.full16 = const_cast<void*>(full_flat16);
  return run_buckets(fn, Kind::kInit, dtype, plan, rank_mask, 0, a, stream);
}

extern "C" zero_status zero_reduce_scatter(const zero_plan* plan, const void* const* grads,
                                           zero_dtype dtype, zero_reduce_op op,
                                           float* const* grad_shards, uint64_t rank_mask,
                                           int64_t bucket_elems, void* stream) {
  const char* fn = "zero_reduce_scatter";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads[r];
    if (in_mask(rank_mask, r)) a.gshard[r] = grad_shards[r];
  }
  set_scale(a, plan->n_ranks, op);
  return run_buckets(fn, Kind::kReduceScatter, dtype, plan, rank_mask, bucket_elems, a, stream);
}

extern "C" zero_status zero_reduce_scatter_range(const zero_plan* plan, const void* const* grads,
                                                 zero_dtype dtype, zero_reduce_op op,
                                                 float* const* grad_shards, uint64_t rank_mask,
                                                 int64_t flat_lo, int64_t flat_hi, void* stream) {
  const char* fn = "zero_reduce_scatter_range";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  if (flat_lo < 0 || flat_hi < flat_lo || flat_hi > plan->padded)
    return fail(ZERO_ERR_INVALID, "%s: range [%" PRId64 ", %" PRId64 ") outside [0, %" PRId64 "]", fn,
                flat_lo, flat_hi, plan->padded);
  ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads[r];
    if (in_mask(rank_mask, r)) a.gshard[r] = grad_shards[r];
  }
  set_scale(a, plan->n_ranks, op);
  set_bounds(a, plan);
  std::vector<Job> jobs;
  build_jobs(plan, rank_mask, flat_lo, flat_hi, jobs);
  if (jobs.empty()) return ZERO_OK;
  a.early = 0;
  return launch_jobs(fn, Kind::kReduceScatter, dtype, a, jobs, stream, nullptr);
}

extern "C" zero_status zero_adamw_shard_step(const zero_plan* plan, float* const* master,
                                             float* const* m, float* const* v,
                                             const float* const* grad_shards,
                                             void* const* out16_shard, zero_dtype dtype,
                                             const zero_adamw_hparams* hp, int64_t step,
                                             uint64_t rank_mask, void* stream) {
  const char* fn = "zero_adamw_shard_step";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  ZERO_TRY(check_hparams(fn, hp, step));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  if (out16_shard) ZERO_TRY(check_ptrs(fn, "out16_shard", out16_shard, plan, rank_mask, true));
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!in_mask(rank_mask, r)) continue;
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
    a.gshard[r] = const_cast<float*>(grad_shards[r]);
    a.shard16[r] = out16_shard ? out16_shard[r] : nullptr;
  }
  a.sc = make_scalars(*hp, step);
  return run_buckets(fn, Kind::kAdamw, dtype, plan, rank_mask, 0, a, stream);
}

extern "C" zero_status zero_cpu_adamw_shard_step(const zero_plan* plan, float* const* master,
                                                 float* const* m, float* const* v,
                                                 const float* const* grad_shards,
                                                 void* const* out16_shard, zero_dtype dtype,
                                                 const zero_adamw_hparams* hp, int64_t step,
                                                 uint64_t rank_mask, int32_t n_threads) {
  const char* fn = "zero_cpu_adamw_shard_step";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  ZERO_TRY(check_hparams(fn, hp, step));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  if (out16_shard) ZERO_TRY(check_ptrs(fn, "out16_shard", out16_shard, plan, rank_mask, true));
  const HostUpdate up{make_scalars(*hp, step), dtype, master, m, v, grad_shards, out16_shard};
  // the masked ranks' shards, concatenated; thread j takes the j-th of nt
  // equal slices of that concatenation
  std::vector<HostPiece> pieces;
  int64_t total = 0;
  try {
    for (int r = 0; r < plan->n_ranks; ++r) {
      if (!in_mask(rank_mask, r) || plan->shard_len[r] == 0) continue;
      pieces.push_back({r, 0, plan->shard_len[r]});
      total += plan->shard_len[r];
    }
  } catch (const std::bad_alloc&) {
    return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  }
  int nt = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  nt = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({nt, kMaxHostThreads,
                                                                (total + 4095) / 4096})));
  auto work = [&](int j) { up.slice(pieces, total * j / nt, total * (j + 1) / nt); };
  std::vector<std::thread> threads;
  try {
    for (int j = 1; j < nt; ++j) threads.emplace_back(work, j);
  } catch (const std::exception&) {
    for (auto& th : threads) th.join();
    return fail(ZERO_ERR_OOM, "%s: could not start host threads", fn);
  }
  work(0);
  for (auto& th : threads) th.join();
  return ZERO_OK;
}

extern "C" zero_status zero_allgather(const zero_plan* plan, const void* const* shards16,
                                      zero_dtype dtype, void* full_flat16, uint64_t rank_mask,
                                      void* stream) {
  const char* fn = "zero_allgather";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  ZERO_TRY(check_ptrs(fn, "shards16", shards16, plan, rank_mask, false));
  if (!full_flat16 && plan->padded > 0)
    return fail(ZERO_ERR_INVALID, "%s: full_flat16 is NULL", fn);
  if (!aligned16(full_flat16)) return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r)
    if (in_mask(rank_mask, r)) a.shard16[r] = const_cast<void*>(shards16[r]);
  a.full16 = full_flat16;
  return run_buckets(fn, Kind::kAllgather, dtype, plan, rank_mask, 0, a, stream);
}

extern "C" zero_status zero_step(const zero_plan* plan, const void* const* grads,
                                 zero_dtype dtype, zero_reduce_op op, float* const* master,
                                 float* const* m, float* const* v, void* full_flat16,
                                 void* const* out16_shard, const zero_adamw_hparams* hp,
                                 int64_t step, uint64_t rank_mask, int64_t bucket_elems,
                                 void* stream) {
  const char* fn = "zero_step";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_hparams(fn, hp, step));
  ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  if (out16_shard) ZERO_TRY(check_ptrs(fn, "out16_shard", out16_shard, plan, rank_mask, true));
  if (full_flat16 && !aligned16(full_flat16))
    return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads[r];
    if (!in_mask(rank_mask, r)) continue;
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
    a.shard16[r] = out16_shard ? out16_shard[r] : nullptr;
  }
  a.full16 = full_flat16;
  a.sc = make_scalars(*hp, step);
  set_scale(a, plan->n_ranks, op);
  return run_buckets(fn, Kind::kStep, dtype, plan, rank_mask, bucket_elems, a, stream);
}

extern "C" zero_status zero_floor_probe(const zero_plan* plan, int32_t kind,
                                        const void* const* grads, zero_dtype dtype,
                                        float* const* master, float* const* m, float* const* v,
                                        void* full_flat16, uint64_t rank_mask,
                                        int64_t bucket_elems, void* stream) {
  const char* fn = "zero_floor_probe";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (kind < 0 || kind > 2) return fail(ZERO_ERR_INVALID, "%s: kind must be 0, 1 or 2", fn);
  ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  if (full_flat16 && !aligned16(full_flat16))
    return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads[r];
    if (!in_mask(rank_mask, r)) continue;
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
  }
  a.full16 = full_flat16;
  a.n_ranks = plan->n_ranks;
  const Kind k = kind == 0 ? Kind::kFloorLaunch : kind == 1 ? Kind::kFloorLoads : Kind::kFloorCopy;
  return run_buckets(fn, k, dtype, plan, rank_mask, bucket_elems, a, stream);
}

extern "C" zero_status zero_amp_init(void* d_state, const zero_amp_config* cfg, void* stream) {
  const char* fn = "zero_amp_init";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_amp_config(fn, cfg));
  if (!d_state) return fail(ZERO_ERR_INVALID, "%s: d_state is NULL", fn);
  if (!aligned16(d_state)) return fail(ZERO_ERR_ALIGN, "%s: d_state is not 16-byte aligned", fn);
  ZERO_TRY(pending_error(fn));
  zero_amp_state init;
  memset(&init, 0, sizeof init);
  init.scale = cfg->init_scale;
  init.hysteresis_left = cfg->hysteresis;
  init.coef = 1.0f;
  const int err = launch_amp_init(static_cast<zero_amp_state*>(d_state), init, stream);
  if (err != 0)
    return fail(ZERO_ERR_CUDA, "%s: launch failed: %s", fn,
                cudaGetErrorString(static_cast<cudaError_t>(err)));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ZERO_OK;
}

extern "C" zero_status zero_amp_workspace_bytes(const zero_plan* plan, uint64_t rank_mask,
                                                int64_t bucket_elems, int64_t* bytes) {
  const char* fn = "zero_amp_workspace_bytes";
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  if (!bytes) return fail(ZERO_ERR_INVALID, "%s: bytes is NULL", fn);
  *bytes = kAmpHeadBytes + count_tiles(plan, rank_mask, bucket_elems) *
                                static_cast<int64_t>(sizeof(NormPartial));
  return ZERO_OK;
}

namespace zero {
namespace {

// Where the mixed-precision step's per-tile sums of squares come from.
enum class AmpStats {
  kReplicas,  // reduce-scatter the replicas into the fp32 shards while summing (k_stats)
  kShards,    // the shards already hold the reduced gradient (k_shard_stats)
  kDone,      // the bucket reductions already wrote every partial (no pass)
};

// The mixed-precision step: the sums of squares as `stats` says, then the
// decision kernel and, unless `decide_only`, the update (k_adamw_amp).
zero_status amp_step(const char* fn, const zero_plan* plan, const void* const* grads,
                     AmpStats stats_from, zero_dtype dtype, zero_reduce_op op,
                     float* const* grad_shards, float* const* master, float* const* m,
                     float* const* v, void* full_flat16, void* const* out16_shard,
                     const zero_adamw_hparams* hp, const zero_amp_config* cfg, void* d_state,
                     void* workspace, int64_t workspace_bytes, uint64_t rank_mask,
                     int64_t bucket_elems, void* stream, bool decide_only = false) {
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_hparams(fn, hp, 1));
  ZERO_TRY(check_amp_config(fn, cfg));
  if (grads) ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, rank_mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, rank_mask, false));
  if (out16_shard) ZERO_TRY(check_ptrs(fn, "out16_shard", out16_shard, plan, rank_mask, true));
  if (full_flat16 && !aligned16(full_flat16))
    return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  if (!d_state) return fail(ZERO_ERR_INVALID, "%s: d_state is NULL", fn);
  if (!aligned16(d_state)) return fail(ZERO_ERR_ALIGN, "%s: d_state is not 16-byte aligned", fn);
  const int64_t tiles = count_tiles(plan, rank_mask, bucket_elems);
  const int64_t need = kAmpHeadBytes + tiles * static_cast<int64_t>(sizeof(NormPartial));
  if (!workspace) return fail(ZERO_ERR_INVALID, "%s: workspace is NULL", fn);
  if (!aligned16(workspace)) return fail(ZERO_ERR_ALIGN, "%s: workspace is not 16-byte aligned", fn);
  if (workspace_bytes < need)
    return fail(ZERO_ERR_INVALID, "%s: workspace holds %" PRId64 " bytes, needs %" PRId64, fn,
                workspace_bytes, need);
  ZERO_TRY(pending_error(fn));
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads ? grads[r] : nullptr;
    if (!in_mask(rank_mask, r)) continue;
    a.gshard[r] = grad_shards[r];
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
    a.shard16[r] = out16_shard ? out16_shard[r] : nullptr;
  }
  a.full16 = full_flat16;
  // workspace: [AmpHead: decision record copies, decision-kernel sums, beta
  // powers, counter][one 16-byte sum of squares per tile]
  AmpHead* head = static_cast<AmpHead*>(workspace);
  a.head = head;
  a.bcast = head->bcast;
  a.partials = reinterpret_cast<NormPartial*>(static_cast<char*>(workspace) + kAmpHeadBytes);
  a.amp_state = static_cast<const zero_amp_state*>(d_state);
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
  set_scale(a, plan->n_ranks, op);
  const Kind stats = stats_from == AmpStats::kReplicas ? Kind::kStats : Kind::kShardStats;
  int64_t done = 0;
  if (stats_from == AmpStats::kDone)
    done = tiles;  // numbered as the bucket reductions numbered them
  else
    ZERO_TRY(run_buckets(fn, stats, dtype, plan, rank_mask, bucket_elems, a, stream, &done));
  if (done == 0) {
    // no owned element: one empty reduction launch still prepares the
    // decision kernel (beta powers, counter)
    a.n_jobs = 0;
    a.n_tiles = 0;
    a.tile_base = 0;
    a.early = 0;
    const int err = launch_kernel(stats, dtype, a, stream);
    if (err != 0)
      return fail(ZERO_ERR_CUDA, "%s: launch failed: %s", fn,
                  cudaGetErrorString(static_cast<cudaError_t>(err)));
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  AmpParams p;
  p.cfg = *cfg;
  p.hp = *hp;
  const int err = launch_amp_finalize(a.partials, done, static_cast<zero_amp_state*>(d_state),
                                      head, p, stream);
  if (err != 0)
    return fail(ZERO_ERR_CUDA, "%s: launch failed: %s", fn,
                cudaGetErrorString(static_cast<cudaError_t>(err)));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (decide_only) return ZERO_OK;
  return run_buckets(fn, Kind::kAdamwAmp, dtype, plan, rank_mask, 0, a, stream);
}

}  // namespace
}  // namespace zero

extern "C" zero_status zero_step_amp(const zero_plan* plan, const void* const* grads,
                                     zero_dtype dtype, zero_reduce_op op,
                                     float* const* grad_shards, float* const* master,
                                     float* const* m, float* const* v, void* full_flat16,
                                     void* const* out16_shard, const zero_adamw_hparams* hp,
                                     const zero_amp_config* cfg, void* d_state, void* workspace,
                                     int64_t workspace_bytes, uint64_t rank_mask,
                                     int64_t bucket_elems, void* stream) {
  const char* fn = "zero_step_amp";
  NvtxRange nvtx_range(fn);
  clear_error();
  if (!grads) return fail(ZERO_ERR_INVALID, "%s: grads is NULL", fn);
  return amp_step(fn, plan, grads, AmpStats::kReplicas, dtype, op, grad_shards, master, m, v,
                  full_flat16, out16_shard, hp, cfg, d_state, workspace, workspace_bytes,
                  rank_mask, bucket_elems, stream);
}

extern "C" zero_status zero_step_amp_shards(const zero_plan* plan, zero_dtype dtype,
                                            float* const* grad_shards, float* const* master,
                                            float* const* m, float* const* v,
                                            void* full_flat16, void* const* out16_shard,
                                            const zero_adamw_hparams* hp,
                                            const zero_amp_config* cfg, void* d_state,
                                            void* workspace, int64_t workspace_bytes,
                                            uint64_t rank_mask, int64_t bucket_elems,
                                            void* stream) {
  const char* fn = "zero_step_amp_shards";
  NvtxRange nvtx_range(fn);
  clear_error();
  return amp_step(fn, plan, nullptr, AmpStats::kShards, dtype, ZERO_REDUCE_SUM, grad_shards,
                  master, m, v, full_flat16, out16_shard, hp, cfg, d_state, workspace,
                  workspace_bytes, rank_mask, bucket_elems, stream);
}

extern "C" zero_status zero_step_amp_reduced(const zero_plan* plan, zero_dtype dtype,
                                             float* const* grad_shards, float* const* master,
                                             float* const* m, float* const* v,
                                             void* full_flat16, void* const* out16_shard,
                                             const zero_adamw_hparams* hp,
                                             const zero_amp_config* cfg, void* d_state,
                                             void* workspace, int64_t workspace_bytes,
                                             uint64_t rank_mask, int64_t bucket_elems,
                                             void* stream) {
  const char* fn = "zero_step_amp_reduced";
  NvtxRange nvtx_range(fn);
  clear_error();
  return amp_step(fn, plan, nullptr, AmpStats::kDone, dtype, ZERO_REDUCE_SUM, grad_shards,
                  master, m, v, full_flat16, out16_shard, hp, cfg, d_state, workspace,
                  workspace_bytes, rank_mask, bucket_elems, stream);
}

extern "C" zero_status zero_reduce_scatter_bucket_amp(
    const zero_plan* plan, const void* const* grads, zero_dtype dtype, zero_reduce_op op,
    float* const* grad_shards, const zero_adamw_hparams* hp, const void* d_state,
    void* workspace, int64_t workspace_bytes, uint64_t rank_mask, int64_t bucket_elems,
    int64_t bucket_index, void* stream) {
  const char* fn = "zero_reduce_scatter_bucket_amp";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_hparams(fn, hp, 1));
  ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, rank_mask, false));
  if (!d_state) return fail(ZERO_ERR_INVALID, "%s: d_state is NULL", fn);
  if (!aligned16(d_state)) return fail(ZERO_ERR_ALIGN, "%s: d_state is not 16-byte aligned", fn);
  const int64_t total = plan->padded;
  const int64_t B = bucket_elems > 0 ? bucket_elems : std::max<int64_t>(total, 1);
  const int64_t n_buckets = (total + B - 1) / B;
  if (bucket_index < 0 || bucket_index >= std::max<int64_t>(n_buckets, 1))
    return fail(ZERO_ERR_INVALID, "%s: bucket %" PRId64 " outside [0, %" PRId64 ")", fn,
                bucket_index, std::max<int64_t>(n_buckets, 1));
  const int64_t need =
      kAmpHeadBytes + count_tiles(plan, rank_mask, bucket_elems) * static_cast<int64_t>(sizeof(NormPartial));
  if (!workspace) return fail(ZERO_ERR_INVALID, "%s: workspace is NULL", fn);
  if (!aligned16(workspace)) return fail(ZERO_ERR_ALIGN, "%s: workspace is not 16-byte aligned", fn);
  if (workspace_bytes < need)
    return fail(ZERO_ERR_INVALID, "%s: workspace holds %" PRId64 " bytes, needs %" PRId64, fn,
                workspace_bytes, need);
  ZERO_TRY(pending_error(fn));
  // the bucket's first tile index: the tiles of the buckets before it, as
  // zero_step_amp numbers them for this mask and bucket size
  std::vector<Job> jobs;
  int64_t base = 0;
  for (int64_t k = 0; k < bucket_index; ++k) {
    build_jobs(plan, rank_mask, k * B, std::min(total, (k + 1) * B), jobs);
    for (const Job& j : jobs) base += (j.len + kTile - 1) / kTile;
  }
  const int64_t lo = bucket_index * B, hi = std::min(total, lo + B);
  build_jobs(plan, rank_mask, lo, hi, jobs);
  if (jobs.empty()) return ZERO_OK;
  ArgsHolder h(new_args());
  if (!h.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  LaunchArgs& a = *h.p;
  for (int r = 0; r < plan->n_ranks; ++r) {
    a.grads[r] = grads[r];
    if (in_mask(rank_mask, r)) a.gshard[r] = grad_shards[r];
  }
  AmpHead* head = static_cast<AmpHead*>(workspace);
  a.head = head;
  a.partials = reinterpret_cast<NormPartial*>(static_cast<char*>(workspace) + kAmpHeadBytes);
  a.amp_state = static_cast<const zero_amp_state*>(d_state);
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
  set_scale(a, plan->n_ranks, op);
  set_bounds(a, plan);
  a.early = 0;
  return launch_jobs(fn, Kind::kStats, dtype, a, jobs, stream, &base);
}

namespace {

// Events reused by zero_zero3_pass and zero_offload_step on this thread
// (created on first use, timing disabled; never destroyed before the thread
// exits).  Re-recording one is safe: a wait already enqueued on it keeps the
// record it saw.
struct EventPool {
  std::vector<cudaEvent_t> ev;
  ~EventPool() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
};

// blocking: events whose cudaEventSynchronize puts the host thread to sleep
// instead of spinning (the offload step's host threads need every core).
zero_status pool_events(const char* fn, size_t n, std::vector<cudaEvent_t>** out,
                        bool blocking = false) {
  static thread_local EventPool spin_pool, block_pool;
  EventPool& pool = blocking ? block_pool : spin_pool;
  while (pool.ev.size() < n) {
    cudaEvent_t e;
    const cudaError_t err = cudaEventCreateWithFlags(
        &e, cudaEventDisableTiming | (blocking ? cudaEventBlockingSync : 0u));
    if (err != cudaSuccess)
      return fail(ZERO_ERR_CUDA, "%s: cudaEventCreateWithFlags: %s", fn, cudaGetErrorString(err));
    pool.ev.push_back(e);
  }
  *out = &pool.ev;
  return ZERO_OK;
}

zero_status cuda_ok(const char* fn, const char* what, cudaError_t e) {
  if (e != cudaSuccess) return fail(ZERO_ERR_CUDA, "%s: %s: %s", fn, what, cudaGetErrorString(e));
  return ZERO_OK;
}

}  // namespace

extern "C" zero_status zero_zero3_pass(const zero_plan* plan, const zero_layer* layers,
                                       int32_t n_layers, void* const* layer_bufs, int32_t n_bufs,
                                       zero_dtype dtype, zero_reduce_op op,
                                       const zero_adamw_hparams* hp, int64_t step,
                                       void* gather_stream, void* step_stream) {
  const char* fn = "zero_zero3_pass";
  NvtxRange nvtx_range(fn);
  clear_error();
  if (!plan) return fail(ZERO_ERR_INVALID, "%s: plan is NULL", fn);
  const uint64_t all = plan->n_ranks >= 64 ? ~UINT64_C(0) : ((UINT64_C(1) << plan->n_ranks) - 1);
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_hparams(fn, hp, step));
  if (!layers || n_layers < 1) return fail(ZERO_ERR_INVALID, "%s: need n_layers >= 1 layers", fn);
  if (!layer_bufs || n_bufs < 1 || n_bufs > 64)
    return fail(ZERO_ERR_INVALID, "%s: need 1 <= n_bufs <= 64 layer buffers", fn);
  for (int32_t b = 0; b < n_bufs; ++b) {
    if (!layer_bufs[b]) return fail(ZERO_ERR_INVALID, "%s: layer_bufs[%d] is NULL", fn, b);
    if (!aligned16(layer_bufs[b])) return fail(ZERO_ERR_ALIGN, "%s: layer_bufs[%d] is not 16-byte aligned", fn, b);
  }
  // every layer's pointers are checked before anything is launched
  for (int32_t l = 0; l < n_layers; ++l) {
    const zero_layer& L = layers[l];
    char msg[1024];
    const zero_status st0 = check_ptrs(fn, "grads", L.grads, plan, all, false, true);
    if (st0 != ZERO_OK) {
      snprintf(msg, sizeof msg, "%s", error_buffer());
      return fail(st0, "%s (layer %d)", msg, l);
    }
    const void* const* per[4] = {reinterpret_cast<const void* const*>(L.master),
                                 reinterpret_cast<const void* const*>(L.m),
                                 reinterpret_cast<const void* const*>(L.v),
                                 reinterpret_cast<const void* const*>(L.shards16)};
    const char* names[4] = {"master", "m", "v", "shards16"};
    for (int k = 0; k < 4; ++k) {
      const zero_status st = check_ptrs(fn, names[k], per[k], plan, all, false);
      if (st != ZERO_OK) {
        snprintf(msg, sizeof msg, "%s", error_buffer());
        return fail(st, "%s (layer %d)", msg, l);
      }
    }
  }
  ZERO_TRY(pending_error(fn));
  std::vector<cudaEvent_t>* ev = nullptr;
  ZERO_TRY(pool_events(fn, static_cast<size_t>(n_bufs) + 2, &ev));
  cudaEvent_t entry = (*ev)[0], gathered = (*ev)[1];
  cudaStream_t gs = static_cast<cudaStream_t>(gather_stream);
  cudaStream_t ss = static_cast<cudaStream_t>(step_stream);
  const bool two = gs != ss;
  if (two) {
    ZERO_TRY(cuda_ok(fn, "cudaEventRecord", cudaEventRecord(entry, ss)));
    ZERO_TRY(cuda_ok(fn, "cudaStreamWaitEvent", cudaStreamWaitEvent(gs, entry, 0)));
  }
  for (int32_t l = 0; l < n_layers; ++l) {
    const zero_layer& L = layers[l];
    cudaEvent_t released = (*ev)[2 + l % n_bufs];
    if (two && l >= n_bufs)
      ZERO_TRY(cuda_ok(fn, "cudaStreamWaitEvent", cudaStreamWaitEvent(gs, released, 0)));
    ZERO_TRY(zero_allgather(plan, L.shards16, dtype, layer_bufs[l % n_bufs], all, gather_stream));
    if (two) {
      ZERO_TRY(cuda_ok(fn, "cudaEventRecord", cudaEventRecord(gathered, gs)));
      ZERO_TRY(cuda_ok(fn, "cudaStreamWaitEvent", cudaStreamWaitEvent(ss, gathered, 0)));
    }
    ZERO_TRY(zero_step(plan, L.grads, dtype, op, L.master, L.m, L.v, nullptr, L.shards16, hp,
                       step, all, 0, step_stream));
    if (two) ZERO_TRY(cuda_ok(fn, "cudaEventRecord", cudaEventRecord(released, ss)));
  }
  return ZERO_OK;
}

namespace {

// How the offload step may touch a buffer: the device writes the fp32
// gradient shards and reads the 16-bit shards across the host link, so those
// must be pinned (or managed) host memory; the host threads read and write
// master/m/v and both shards, so none of them may be device memory.
zero_status check_host_buffers(const char* fn, const char* what, void* const* arr,
                               const zero_plan* plan, uint64_t mask, bool device_accessible) {
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!in_mask(mask, r) || plan->shard_len[r] == 0) continue;
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, arr[r]);
    if (e != cudaSuccess)
      return fail(ZERO_ERR_CUDA, "%s: cudaPointerGetAttributes(%s[%d]): %s", fn, what, r,
                  cudaGetErrorString(e));
    const bool pinned = at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged;
    if (device_accessible && !pinned)
      return fail(ZERO_ERR_INVALID, "%s: %s[%d] must be pinned (or managed) host memory", fn,
                  what, r);
    if (at.type == cudaMemoryTypeDevice)
      return fail(ZERO_ERR_INVALID, "%s: %s[%d] is device memory; the host updates it", fn,
                  what, r);
  }
  return ZERO_OK;
}

// The checks both offload steps make after the plain argument checks: the
// stream is not capturing (the host waits for the device), the buffers are
// where the host and the device can reach them, and the chunking is bounded.
zero_status check_offload(const char* fn, const zero_plan* plan, uint64_t mask,
                          float* const* grad_shards, float* const* master, float* const* m,
                          float* const* v, void* const* out16_shard, void* full_flat16,
                          int64_t chunk_elems, void* stream, int64_t* C, int64_t* K) {
  ZERO_TRY(check_ptrs(fn, "grad_shards", grad_shards, plan, mask, false));
  ZERO_TRY(check_ptrs(fn, "master", master, plan, mask, false));
  ZERO_TRY(check_ptrs(fn, "m", m, plan, mask, false));
  ZERO_TRY(check_ptrs(fn, "v", v, plan, mask, false));
  ZERO_TRY(check_ptrs(fn, "out16_shard", out16_shard, plan, mask, false));
  if (full_flat16 && !aligned16(full_flat16))
    return fail(ZERO_ERR_ALIGN, "%s: full_flat16 is not 16-byte aligned", fn);
  const int64_t total = plan->padded;
  *C = chunk_elems > 0 ? chunk_elems : std::max<int64_t>(total, 1);
  *K = (total + *C - 1) / *C;
  if (*K > kMaxOffloadChunks)
    return fail(ZERO_ERR_INVALID, "%s: %" PRId64 " chunks of %" PRId64 " elements; at most %d",
                fn, *K, *C, kMaxOffloadChunks);
  ZERO_TRY(pending_error(fn));
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  ZERO_TRY(cuda_ok(fn, "cudaStreamIsCapturing",
                   cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap)));
  if (cap != cudaStreamCaptureStatusNone)
    return fail(ZERO_ERR_UNSUPPORTED, "%s: cannot be captured: the host waits for the device", fn);
  ZERO_TRY(check_host_buffers(fn, "grad_shards", reinterpret_cast<void* const*>(grad_shards),
                              plan, mask, true));
  ZERO_TRY(check_host_buffers(fn, "out16_shard", out16_shard, plan, mask, true));
  ZERO_TRY(check_host_buffers(fn, "master", reinterpret_cast<void* const*>(master), plan, mask,
                              false));
  ZERO_TRY(check_host_buffers(fn, "m", reinterpret_cast<void* const*>(m), plan, mask, false));
  ZERO_TRY(check_host_buffers(fn, "v", reinterpret_cast<void* const*>(v), plan, mask, false));
  return ZERO_OK;
}

// Launch `kind` over the masked ranks' elements of the flat range [lo, hi),
// ordered after everything before it on the stream.
zero_status launch_range(const char* fn, Kind kind, zero_dtype dtype, const zero_plan* plan,
                         uint64_t mask, int64_t lo, int64_t hi, LaunchArgs& a, void* stream) {
  std::vector<Job> jobs;
  build_jobs(plan, mask, lo, hi, jobs);
  if (jobs.empty()) return ZERO_OK;
  a.early = 0;
  return launch_jobs(fn, kind, dtype, a, jobs, stream, nullptr);
}

// The host side of the offload pipeline: chunk k's update may start once
// `ready` exceeds k; each worker counts itself into done[k] when its share of
// chunk k is written.
struct OffloadSync {
  std::mutex mu;
  std::condition_variable ready_cv, done_cv;
  int64_t ready = 0;
  bool abort = false;
  std::vector<int> done;
};

// The host update of every chunk of C flat elements (K chunks) by n_threads
// workers, each chunk's gather into full_flat16 (nullable) enqueued on
// `stream` as soon as the workers have written it.  Chunk k is released to
// the workers when event ev[k] has completed (n_events == K), all chunks when
// ev[0] has (n_events == 1), or at once (n_events == 0).
zero_status host_update_pipeline(const char* fn, const zero_plan* plan, uint64_t mask,
                                 zero_dtype dtype, const HostUpdate& up, int64_t C, int64_t K,
                                 const std::vector<cudaEvent_t>* ev, int64_t n_events,
                                 void* const* out16_shard, void* full_flat16,
                                 int32_t n_threads, void* stream) {
  const int64_t total = plan->padded;
  // each chunk's host pieces: the masked ranks' runs cut to the chunk
  std::vector<std::vector<HostPiece>> pieces;
  std::vector<int64_t> chunk_len;
  OffloadSync sync;
  try {
    pieces.resize(static_cast<size_t>(K));
    chunk_len.assign(static_cast<size_t>(K), 0);
    sync.done.assign(static_cast<size_t>(K), 0);
    for (int64_t k = 0; k < K; ++k) {
      const int64_t lo = k * C, hi = std::min(total, lo + C);
      for (int r = 0; r < plan->n_ranks; ++r) {
        if (!in_mask(mask, r)) continue;
        for (const auto& run : plan->runs[r]) {
          const int64_t a = std::max(lo, run.flat_off);
          const int64_t b = std::min(hi, run.flat_off + run.len);
          if (a >= b) continue;
          pieces[k].push_back({r, run.shard_off + (a - run.flat_off), b - a});
          chunk_len[k] += b - a;
        }
      }
    }
  } catch (const std::bad_alloc&) {
    return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  }
  ArgsHolder gat(new_args());
  if (!gat.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  for (int r = 0; r < plan->n_ranks; ++r)
    if (in_mask(mask, r)) gat.p->shard16[r] = out16_shard[r];
  gat.p->full16 = full_flat16;
  set_bounds(*gat.p, plan);
  if (n_events == 0) sync.ready = K;

  // the calling thread waits for the device and launches the gathers, so by
  // default one hardware thread is left to it
  int nt = n_threads > 0 ? n_threads
                         : static_cast<int>(std::thread::hardware_concurrency()) - 1;
  nt = std::max(1, std::min(nt, kMaxHostThreads));
  auto worker = [&](int j) {
    for (int64_t k = 0; k < K; ++k) {
      {
        std::unique_lock<std::mutex> lk(sync.mu);
        sync.ready_cv.wait(lk, [&] { return sync.ready > k || sync.abort; });
        if (sync.abort) return;
      }
      const int64_t T = chunk_len[k];
      up.slice(pieces[k], T * j / nt, T * (j + 1) / nt);
      std::lock_guard<std::mutex> lk(sync.mu);
      if (++sync.done[k] == nt) sync.done_cv.notify_all();
    }
  };
  std::vector<std::thread> threads;
  auto stop = [&](zero_status st) {
    {
      std::lock_guard<std::mutex> lk(sync.mu);
      sync.abort = true;
    }
    sync.ready_cv.notify_all();
    for (auto& th : threads) th.join();
    return st;
  };
  try {
    for (int j = 0; j < nt; ++j) threads.emplace_back(worker, j);
  } catch (const std::exception&) {
    return stop(fail(ZERO_ERR_OOM, "%s: could not start host threads", fn));
  }

  // release the chunks as their events complete; gather every chunk the
  // workers have finished, as soon as it is finished
  int64_t gathered = 0;
  auto gather_finished = [&](bool wait_all) -> zero_status {
    while (gathered < K) {
      {
        std::unique_lock<std::mutex> lk(sync.mu);
        if (wait_all)
          sync.done_cv.wait(lk, [&] { return sync.done[gathered] == nt; });
        else if (sync.done[gathered] != nt)
          return ZERO_OK;
      }
      const int64_t lo = gathered * C, hi = std::min(total, lo + C);
      if (full_flat16) {
        const zero_status st = launch_range(fn, Kind::kAllgather, dtype, plan, mask, lo, hi,
                                            *gat.p, stream);
        if (st != ZERO_OK) return st;
      }
      ++gathered;
    }
    return ZERO_OK;
  };
  for (int64_t k = 0; k < n_events; ++k) {
    const cudaError_t e = cudaEventSynchronize((*ev)[k]);
    if (e != cudaSuccess)
      return stop(fail(ZERO_ERR_CUDA, "%s: device work before chunk %" PRId64 ": %s", fn, k,
                       cudaGetErrorString(e)));
    {
      std::lock_guard<std::mutex> lk(sync.mu);
      sync.ready = n_events == K ? k + 1 : K;
    }
    sync.ready_cv.notify_all();
    const zero_status st = gather_finished(false);
    if (st != ZERO_OK) return stop(st);
  }
  const zero_status st = gather_finished(true);
  if (st != ZERO_OK) return stop(st);
  for (auto& th : threads) th.join();
  return ZERO_OK;
}

}  // namespace

extern "C" zero_status zero_offload_step(const zero_plan* plan, const void* const* grads,
                                         zero_dtype dtype, zero_reduce_op op,
                                         float* const* grad_shards, float* const* master,
                                         float* const* m, float* const* v,
                                         void* const* out16_shard, void* full_flat16,
                                         const zero_adamw_hparams* hp, int64_t step,
                                         uint64_t rank_mask, int64_t chunk_elems,
                                         int32_t n_threads, void* stream) {
  const char* fn = "zero_offload_step";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  ZERO_TRY(check_dtype(fn, dtype));
  if (op != ZERO_REDUCE_SUM && op != ZERO_REDUCE_AVG) return fail(ZERO_ERR_INVALID, "%s: unknown reduce op", fn);
  ZERO_TRY(check_hparams(fn, hp, step));
  if (grads) ZERO_TRY(check_ptrs(fn, "grads", grads, plan, rank_mask, false, true));
  int64_t C = 0, K = 0;
  ZERO_TRY(check_offload(fn, plan, rank_mask, grad_shards, master, m, v, out16_shard,
                         full_flat16, chunk_elems, stream, &C, &K));
  if (K == 0) return ZERO_OK;
  const int64_t total = plan->padded;

  // every chunk's reduction, each followed by its event; without grads (the
  // shards already hold the reduced gradients) one event marks the end of
  // the work enqueued on the stream before the call
  ArgsHolder red(new_args());
  if (!red.p) return fail(ZERO_ERR_OOM, "%s: out of host memory", fn);
  for (int r = 0; r < plan->n_ranks; ++r) {
    red.p->grads[r] = grads ? grads[r] : nullptr;
    if (in_mask(rank_mask, r)) red.p->gshard[r] = grad_shards[r];
  }
  set_scale(*red.p, plan->n_ranks, op);
  set_bounds(*red.p, plan);
  std::vector<cudaEvent_t>* ev = nullptr;
  const int64_t n_events = grads ? K : 1;
  ZERO_TRY(pool_events(fn, static_cast<size_t>(n_events), &ev, true));
  for (int64_t k = 0; k < n_events; ++k) {
    if (grads) {
      const int64_t lo = k * C, hi = std::min(total, lo + C);
      ZERO_TRY(launch_range(fn, Kind::kReduceScatter, dtype, plan, rank_mask, lo, hi, *red.p,
                            stream));
    }
    ZERO_TRY(cuda_ok(fn, "cudaEventRecord",
                     cudaEventRecord((*ev)[k], static_cast<cudaStream_t>(stream))));
  }
  const HostUpdate up{make_scalars(*hp, step), dtype, master, m, v, grad_shards, out16_shard};
  return host_update_pipeline(fn, plan, rank_mask, dtype, up, C, K, ev, n_events, out16_shard,
                              full_flat16, n_threads, stream);
}

extern "C" zero_status zero_offload_step_amp(
    const zero_plan* plan, const void* const* grads, zero_dtype dtype, zero_reduce_op op,
    float* const* grad_shards, float* const* master, float* const* m, float* const* v,
    void* const* out16_shard, void* full_flat16, const zero_adamw_hparams* hp,
    const zero_amp_config* cfg, void* d_state, void* workspace, int64_t workspace_bytes,
    uint64_t rank_mask, int64_t bucket_elems, int64_t chunk_elems, int32_t n_threads,
    void* stream) {
  const char* fn = "zero_offload_step_amp";
  NvtxRange nvtx_range(fn);
  clear_error();
  ZERO_TRY(check_plan_mask(fn, plan, rank_mask));
  int64_t C = 0, K = 0;
  ZERO_TRY(check_offload(fn, plan, rank_mask, grad_shards, master, m, v, out16_shard,
                         full_flat16, chunk_elems, stream, &C, &K));
  // the sums of squares (from the replicas, or already in the workspace) and
  // the decision kernel; amp_step checks its own arguments before launching
  ZERO_TRY(amp_step(fn, plan, grads, grads ? AmpStats::kReplicas : AmpStats::kDone, dtype, op,
                    grad_shards, master, m, v, full_flat16, out16_shard, hp, cfg, d_state,
                    workspace, workspace_bytes, rank_mask, bucket_elems, stream, true));
  // the host reads the decision
  zero_amp_state st;
  std::vector<cudaEvent_t>* ev = nullptr;
  ZERO_TRY(pool_events(fn, 1, &ev, true));
  ZERO_TRY(cuda_ok(fn, "cudaMemcpyAsync",
                   cudaMemcpyAsync(&st, d_state, sizeof st, cudaMemcpyDeviceToHost,
                                   static_cast<cudaStream_t>(stream))));
  ZERO_TRY(cuda_ok(fn, "cudaEventRecord",
                   cudaEventRecord((*ev)[0], static_cast<cudaStream_t>(stream))));
  ZERO_TRY(cuda_ok(fn, "cudaEventSynchronize", cudaEventSynchronize((*ev)[0])));
  if (st.overflow != 0 || K == 0) return ZERO_OK;  // skipped: nothing changes
  HostUpdate up{StepScalars{}, dtype, master, m, v, grad_shards, out16_shard};
  up.sc = StepScalars{st.sc[0], st.sc[1], st.sc[2], st.sc[3], st.sc[4], st.sc[5], st.sc[6],
                      st.sc[7]};
  up.scaled = true;
  up.coef = st.coef;
  return host_update_pipeline(fn, plan, rank_mask, dtype, up, C, K, nullptr, 0, out16_shard,
                              full_flat16, n_threads, stream);
}

extern "C" zero_status zero_sync(void* stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ZERO_ERR_CUDA, "zero_sync: %s", cudaGetErrorString(e));
  const int dev_err = take_device_error(stream);
  if (dev_err == kErrBounds)
    return fail(ZERO_ERR_INVALID, "zero_sync: a kernel index fell outside its buffer "
                                  "(bounds-checked build)");
  if (dev_err)
    return fail(ZERO_ERR_TIMEOUT, "zero_sync: a kernel gave up a bounded wait on the device");
  return ZERO_OK;
}

extern "C" zero_status zero_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  const char* fn = "zero_selftest_wait_timeout";
  clear_error();
  if (limit_ns < 1000 || limit_ns > INT64_C(10000000000))
    return fail(ZERO_ERR_INVALID, "%s: limit_ns must lie in [1e3, 1e10]", fn);
  ZERO_TRY(pending_error(fn));
  const int err = launch_selftest_wait(limit_ns, stream);
  if (err != 0)
    return fail(ZERO_ERR_CUDA, "%s: launch failed: %s", fn,
                cudaGetErrorString(static_cast<cudaError_t>(err)));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ZERO_OK;
}

extern "C" const char* zero_last_error(void) { return error_buffer(); }

extern "C" int64_t zero_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char* zero_version(void) { return "zero-gb300 0.1.0 (sm_103a)"; }
