// Partition plan and memory model of the ZeRO sharded optimizer step (host).
//
// Flat mode follows "DeepSpeed ZeRO-2 ... DeepSpeedZeroOptimizer"
// (discosf.com) §2.1 / §4.1: the group is flattened into one contiguous
// buffer and cut into as many near-equal partitions as there are ranks.  This
// library reads "near-equal" as equal partitions of S elements, with the flat
// buffer padded at its tail to a multiple of n_ranks * align_elems; tensors
// follow one another with no gap.
//
// Round-robin mode follows "ZeRO 优化器" (cookllm.com), 参数分配策略: tensor
// i of named_parameters() belongs whole to rank i % world_size; the shard of
// a rank packs its tensors in increasing i.
#include <inttypes.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>

#include "zero_capi_util.h"
#include "zero_internal.h"

namespace {

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Runs: merge consecutive segments that continue each other in both the flat
// and the shard index space.
void build_runs(zero_plan* p) {
  p->runs.assign(p->n_ranks, {});
  for (int r = 0; r < p->n_ranks; ++r) {
    auto& out = p->runs[r];
    for (const auto& s : p->segs[r]) {
      if (!out.empty() && out.back().flat_off + out.back().len == s.flat_off &&
          out.back().shard_off + out.back().len == s.shard_off) {
        out.back().len += s.len;
      } else {
        out.push_back({s.flat_off, s.shard_off, s.len});
      }
    }
  }
}

}  // namespace

extern "C" zero_status zero_plan_partitions(const int64_t* numel, int32_t n_tensors,
                                            int32_t n_ranks, zero_part_mode mode,
                                            int32_t align_elems, zero_plan** out) {
  using zero::fail;
  zero::clear_error();
  if (!out) return fail(ZERO_ERR_INVALID, "zero_plan_partitions: out is NULL");
  *out = nullptr;
  if (!numel) return fail(ZERO_ERR_INVALID, "zero_plan_partitions: numel is NULL");
  if (n_tensors < 1) return fail(ZERO_ERR_INVALID, "zero_plan_partitions: n_tensors < 1");
  if (n_ranks < 1 || n_ranks > zero::kMaxRanks)
    return fail(ZERO_ERR_INVALID, "zero_plan_partitions: n_ranks must be in [1, 64]");
  if (mode != ZERO_PART_FLAT && mode != ZERO_PART_ROUND_ROBIN)
    return fail(ZERO_ERR_INVALID, "zero_plan_partitions: unknown partition mode");
  if (mode == ZERO_PART_FLAT && (!is_pow2(align_elems) || align_elems > 4096))
    return fail(ZERO_ERR_INVALID,
                "zero_plan_partitions: align_elems must be a power of two in [1, 4096]");

  zero_plan* p = new (std::nothrow) zero_plan();
  if (!p) return fail(ZERO_ERR_OOM, "zero_plan_partitions: out of host memory");
  try {
    p->n_ranks = n_ranks;
    p->mode = mode;
    p->align = mode == ZERO_PART_FLAT ? align_elems : 1;
    p->numel.assign(numel, numel + n_tensors);
    p->tensor_start.resize(n_tensors);
    const int64_t limit = INT64_C(1) << 56;  // keeps every offset and byte count in int64
    int64_t total = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
      if (numel[k] < 0 || numel[k] > limit - total) {
        delete p;
        return fail(ZERO_ERR_INVALID, "zero_plan_partitions: numel[%d] = %" PRId64
                    " is negative or the group is too large", k, numel[k]);
      }
      p->tensor_start[k] = total;
      total += numel[k];
    }
    p->phi = total;
    p->segs.assign(n_ranks, {});
    p->shard_len.assign(n_ranks, 0);
    p->shard_flat.assign(n_ranks, -1);

    if (mode == ZERO_PART_FLAT) {
      const int64_t unit = static_cast<int64_t>(n_ranks) * align_elems;
      p->padded = (total + unit - 1) / unit * unit;
      const int64_t S = p->padded / n_ranks;
      // walk tensors once; each rank's range [r*S, (r+1)*S) collects the
      // pieces of the tensors it overlaps, then the padding.
      for (int32_t r = 0; r < n_ranks; ++r) {
        const int64_t lo = r * S, hi = lo + S;
        p->shard_len[r] = S;
        p->shard_flat[r] = lo;
        // first tensor whose end lies past lo
        auto it = std::upper_bound(p->tensor_start.begin(), p->tensor_start.end(), lo);
        int32_t k = static_cast<int32_t>(it - p->tensor_start.begin()) - 1;
        if (k < 0) k = 0;
        for (; k < n_tensors && p->tensor_start[k] < hi; ++k) {
          const int64_t a = std::max(lo, p->tensor_start[k]);
          const int64_t b = std::min(hi, p->tensor_start[k] + numel[k]);
          if (a < b) p->segs[r].push_back({k, a - p->tensor_start[k], a, a - lo, b - a});
        }
        if (total < hi) {
          const int64_t a = std::max(lo, total);
          p->segs[r].push_back({-1, 0, a, a - lo, hi - a});
        }
      }
    } else {
      p->padded = total;
      for (int32_t k = 0; k < n_tensors; ++k) {
        const int32_t r = k % n_ranks;
        if (numel[k] > 0)
          p->segs[r].push_back({k, 0, p->tensor_start[k], p->shard_len[r], numel[k]});
        p->shard_len[r] += numel[k];
      }
    }
    build_runs(p);
  } catch (const std::bad_alloc&) {
    delete p;
    return fail(ZERO_ERR_OOM, "zero_plan_partitions: out of host memory");
  }
  *out = p;
  return ZERO_OK;
}

extern "C" void zero_plan_destroy(zero_plan* plan) { delete plan; }

extern "C" zero_status zero_plan_total(const zero_plan* plan, int64_t* phi, int64_t* padded) {
  zero::clear_error();
  if (!plan || !phi || !padded) return zero::fail(ZERO_ERR_INVALID, "zero_plan_total: NULL argument");
  *phi = plan->phi;
  *padded = plan->padded;
  return ZERO_OK;
}

extern "C" zero_status zero_plan_info(const zero_plan* plan, int32_t* n_ranks, int32_t* mode,
                                      int32_t* align_elems, int32_t* n_tensors) {
  zero::clear_error();
  if (!plan || !n_ranks || !mode || !align_elems || !n_tensors)
    return zero::fail(ZERO_ERR_INVALID, "zero_plan_info: NULL argument");
  *n_ranks = plan->n_ranks;
  *mode = plan->mode;
  *align_elems = plan->align;
  *n_tensors = static_cast<int32_t>(plan->numel.size());
  return ZERO_OK;
}

extern "C" zero_status zero_plan_shard(const zero_plan* plan, int32_t rank, int64_t* flat_off,
                                       int64_t* len) {
  zero::clear_error();
  if (!plan || !flat_off || !len) return zero::fail(ZERO_ERR_INVALID, "zero_plan_shard: NULL argument");
  if (rank < 0 || rank >= plan->n_ranks)
    return zero::fail(ZERO_ERR_INVALID, "zero_plan_shard: rank %d out of range", rank);
  *flat_off = plan->shard_flat[rank];
  *len = plan->shard_len[rank];
  return ZERO_OK;
}

extern "C" zero_status zero_plan_segments(const zero_plan* plan, int32_t rank,
                                          int64_t* tensor_idx, int64_t* tensor_off,
                                          int64_t* flat_off, int64_t* shard_off, int64_t* len,
                                          int64_t cap, int64_t* n_out) {
  zero::clear_error();
  if (!plan || !n_out) return zero::fail(ZERO_ERR_INVALID, "zero_plan_segments: NULL argument");
  if (rank < 0 || rank >= plan->n_ranks)
    return zero::fail(ZERO_ERR_INVALID, "zero_plan_segments: rank %d out of range", rank);
  if (cap < 0) return zero::fail(ZERO_ERR_INVALID, "zero_plan_segments: cap < 0");
  if (cap > 0 && (!tensor_idx || !tensor_off || !flat_off || !shard_off || !len))
    return zero::fail(ZERO_ERR_INVALID, "zero_plan_segments: NULL output array");
  const auto& segs = plan->segs[rank];
  const int64_t n = static_cast<int64_t>(segs.size());
  for (int64_t j = 0; j < std::min(n, cap); ++j) {
    tensor_idx[j] = segs[j].tensor;
    tensor_off[j] = segs[j].tensor_off;
    flat_off[j] = segs[j].flat_off;
    shard_off[j] = segs[j].shard_off;
    len[j] = segs[j].len;
  }
  *n_out = n;
  return ZERO_OK;
}

extern "C" zero_status zero_plan_describe(const zero_plan* plan, char* buf, int64_t cap) {
  zero::clear_error();
  if (!plan || !buf || cap < 1) return zero::fail(ZERO_ERR_INVALID, "zero_plan_describe: bad argument");
  std::string s;
  char line[256];
  snprintf(line, sizeof line,
           "zero_plan mode=%s n_ranks=%d align=%d tensors=%zu phi=%" PRId64 " padded=%" PRId64 "\n",
           plan->mode == ZERO_PART_FLAT ? "flat" : "round_robin", plan->n_ranks, plan->align,
           plan->numel.size(), plan->phi, plan->padded);
  s += line;
  for (int r = 0; r < plan->n_ranks; ++r) {
    snprintf(line, sizeof line,
             "  rank %d: shard_len=%" PRId64 " flat_off=%" PRId64 " segments=%zu runs=%zu\n", r,
             plan->shard_len[r], plan->shard_flat[r], plan->segs[r].size(), plan->runs[r].size());
    s += line;
  }
  const size_t n = std::min<size_t>(s.size(), static_cast<size_t>(cap - 1));
  memcpy(buf, s.data(), n);
  buf[n] = '\0';
  return ZERO_OK;
}

// Per-rank model-state bytes for stage 0..3 of mixed-precision Adam:
// 2 B of 16-bit parameters, 2 B of 16-bit gradients and 12 B of fp32
// master + m + v per element, each either held whole or split N ways
// ("ZeRO / DeepSpeed 深度解读报告" §3.3; "ZeRO 优化器" stage tables).
extern "C" zero_status zero_memory_bytes(int32_t stage, int64_t phi, int32_t n_ranks,
                                         int64_t* num, int64_t* den) {
  zero::clear_error();
  if (!num || !den) return zero::fail(ZERO_ERR_INVALID, "zero_memory_bytes: NULL output");
  if (phi < 0 || n_ranks < 1) return zero::fail(ZERO_ERR_INVALID, "zero_memory_bytes: phi < 0 or n_ranks < 1");
  static const int64_t kWhole[4] = {16, 4, 2, 0};   // bytes per element kept on every rank
  static const int64_t kSplit[4] = {0, 12, 14, 16};  // bytes per element split over ranks
  if (stage < 0 || stage > 3) return zero::fail(ZERO_ERR_INVALID, "zero_memory_bytes: stage must be 0..3");
  // whole*phi + split*phi/N  ==  (whole*phi*N + split*phi) / N
  __int128 a = static_cast<__int128>(kWhole[stage]) * phi * n_ranks +
               static_cast<__int128>(kSplit[stage]) * phi;
  __int128 b = n_ranks;
  __int128 x = a, y = b;
  while (y != 0) {
    __int128 t = x % y;
    x = y;
    y = t;
  }
  if (x > 1) {
    a /= x;
    b /= x;
  }
  if (a > INT64_MAX) return zero::fail(ZERO_ERR_INVALID, "zero_memory_bytes: result overflows int64");
  *num = static_cast<int64_t>(a);
  *den = static_cast<int64_t>(b);
  return ZERO_OK;
}
