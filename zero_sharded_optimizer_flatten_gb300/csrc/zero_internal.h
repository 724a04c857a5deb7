// Internal structures shared by the host launcher and the CUDA kernels of the
// ZeRO sharded optimizer step.  Not part of the public ABI (include/zero.h).
#pragma once

#include <stdint.h>

#include <string>
#include <vector>

#include "zero.h"

namespace zero {

constexpr int kMaxRanks = 64;     // rank_mask is a uint64_t
#ifndef ZERO_THREADS
#define ZERO_THREADS 256
#endif
constexpr int kThreads = ZERO_THREADS;  // threads per CTA of every kernel
constexpr int kVec = 4;           // elements per quad (8 B of 16-bit, 16 B of fp32 data)
constexpr int kHalf = kThreads * kVec;  // 1024: distance between a thread's two quads
constexpr int kTile = 2 * kHalf;  // 2048 elements per CTA per tile
constexpr int kMaxJobs = 192;     // jobs carried in one launch's parameters

// Resident CTAs per SM the kernels are compiled for (caps registers at 64),
// and the grid: ZERO_GRID_MULT = 0 launches one CTA per tile; k > 0 caps the
// grid at k times the resident capacity (the CTAs then stride over tiles).
// Measured on the BERT-base group (8 replicas): one CTA per tile 6931 GB/s,
// 32x 6868, 8x 6567, 1x (persistent) 6158 -- the hardware's CTA scheduler
// spreads the concurrently open DRAM streams better than a grid stride does.
#ifndef ZERO_MIN_BLOCKS
#define ZERO_MIN_BLOCKS 4
#endif
#ifndef ZERO_GRID_MULT
#define ZERO_GRID_MULT 0
#endif
// Consecutive 2048-element tiles one CTA of the all-gather copies.  Measured
// (zero_allgather of every shard): LLaMA-7B group 6421 / 7199 / 7156 / 7167
// GB/s for 1 / 2 / 4 / 8 tiles, BERT-base 5919 / 6783 / 6600 / 6640, one
// LLaMA-13B MLP layer 6250 / 6975 / 6841 / 6841.
#ifndef ZERO_GATHER_TILES
#define ZERO_GATHER_TILES 2
#endif
constexpr int kGatherTiles = ZERO_GATHER_TILES;

// The shard-only sum of squares (k_shard_stats) gives a 2048-element tile to
// kShardStatsThreads threads, each holding four of the tile's 256 slots, so
// a CTA takes kShardStatsTiles consecutive tiles.
constexpr int kShardStatsThreads = 64;
constexpr int kShardStatsTiles = kThreads / kShardStatsThreads;
static_assert(kTile / kVec / 2 == 4 * kShardStatsThreads, "four slots per thread");

// Bounds-checked build: every kernel access is checked against the plan's
// buffer lengths; a violation skips the access and sets the device error
// word to 2 (zero_sync reports it).
#ifndef ZERO_DEBUG_BOUNDS
#define ZERO_DEBUG_BOUNDS 0
#endif
constexpr int kErrTimeout = 1;
constexpr int kErrBounds = 2;

// 256-byte L2 prefetch hints on the streaming loads (tuning switch).
#ifndef ZERO_L2_PREFETCH
#define ZERO_L2_PREFETCH 0
#endif

// Binary32 constants of one AdamW step, formed on the host in binary64 and
// rounded once each (see zero_adamw_hparams).
struct StepScalars {
  float d, b1, b2, c1, c2, ss, sb, eps;
};

// How the rank-ordered sum becomes the gradient: kept (SUM), multiplied by the
// exact power of two 1/N, or divided by N.  Multiplying by an exact 1/N and
// dividing by N round the same real number, so both give the binary32
// quotient of the sum by N.
enum ScaleMode : int32_t { kScaleNone = 0, kScaleMul = 1, kScaleDiv = 2 };

// A contiguous run of one rank's elements: flat indices
// [flat_off, flat_off + len) map to shard indices [shard_off, shard_off + len).
// vec != 0: flat_off, shard_off and len are multiples of kVec, so the run is
// processed in quads (8-byte 16-bit and 16-byte fp32 accesses); otherwise
// element by element.
struct Job {
  int64_t flat_off;
  int64_t shard_off;
  int64_t len;
  int64_t tile_begin;  // index of the job's first tile in the launch
  int32_t rank;
  int32_t vec;
};

// Parameters of one launch.  Passed by value as a __grid_constant__ kernel
// parameter (about 10 KB), so the job table needs no device allocation.
struct LaunchArgs {
  const void* grads[kMaxRanks];  // 16-bit flat replicas (reduce/step)
  float* master[kMaxRanks];
  float* m[kMaxRanks];
  float* v[kMaxRanks];
  float* gshard[kMaxRanks];        // fp32 reduced gradient shards (adamw in / reduce out)
  void* shard16[kMaxRanks];        // 16-bit shard buffers (nullable entries)
  void* full16;                    // gathered flat 16-bit buffer (nullable)
  StepScalars sc;
  float inv_n;                     // 1/N when N is a power of two
  float n_f;                       // N as binary32
  int32_t scale_mode;
  int32_t n_ranks;                 // gradient replicas summed
  int32_t n_jobs;
  int32_t early;                   // launched early: wait for the previous launch at the end
  int64_t n_tiles;
  struct NormPartial* partials;    // mixed-precision: per-tile sums of squares
  int64_t tile_base;               // index of this launch's first tile among the step's
  const struct AmpBcast* bcast;    // mixed-precision: copies of the decision record
  struct AmpHead* head;            // mixed-precision: workspace head (reduction writes)
  const zero_amp_state* amp_state; // mixed-precision: the device state (step count)
  double beta1, beta2;             // mixed-precision: AdamW betas
  int* err;                        // device error word (bounded wait, bounds check)
  int64_t flat_len;                // bounds-checked builds: length of the flat buffers
  int64_t shard_len[kMaxRanks];    // bounds-checked builds: shard lengths
  Job jobs[kMaxJobs];
};

enum class Kind {
  kStep, kReduceScatter, kAdamw, kAllgather, kInit, kStats, kShardStats, kAdamwAmp,
  kFloorLaunch, kFloorLoads, kFloorCopy  // measurement floors of kStep (zero_floor_probe)
};

// The decision of a mixed-precision step as the update kernel needs it.  The
// decision kernel writes kAmpCopies copies, 64 bytes apart, at the start of
// the workspace; CTA b reads copy b % kAmpCopies with one thread, so the
// tens of thousands of CTAs of the update do not all hit one L2 line.
struct alignas(16) AmpBcast {
  int32_t overflow;
  float coef;
  int32_t pad_[2];
  float sc[8];
  int32_t pad2_[4];
};
static_assert(sizeof(AmpBcast) == 64, "one copy per 64-byte line segment");
constexpr int kAmpCopies = 64;

// One tile's sum of squared gradients as two unevaluated sums of binary32
// pairs: a = squares below 2^64, b = the others times 2^-64 (exact scaling),
// so that no partial sum of finite squares can overflow binary32.  The
// tile's sum is (a_hi + a_lo) + 2^64 (b_hi + b_lo).
struct alignas(16) NormPartial {
  float a_hi, a_lo, b_hi, b_lo;
};
static_assert(sizeof(NormPartial) == 16, "one 16-byte store per tile");

// The decision kernel's CTAs (each sums a share of the per-tile partials;
// the last one to finish adds the CTAs' sums and decides) and their threads.
constexpr int kFinCtas = 32;
constexpr int kFinThreads = 256;

// Head of the mixed-precision workspace; the per-tile partials follow it.
struct alignas(64) AmpHead {
  AmpBcast bcast[kAmpCopies];        // the decision record, kAmpCopies times
  NormPartial cta_part[kFinCtas];    // the decision kernel's per-CTA sums
  double beta_pow[2];                // beta1^t and beta2^t of the step t = step + 1
  int32_t arrived;                   // decision-kernel CTAs done (reset every step)
};
constexpr int64_t kAmpHeadBytes = 8192;
static_assert(sizeof(AmpHead) <= kAmpHeadBytes, "workspace head");

// Parameters of the decision kernel of the mixed-precision step.
struct AmpParams {
  zero_amp_config cfg;
  zero_adamw_hparams hp;
};

// The binary32 constants of step t (zero_capi.cpp).
StepScalars make_scalars(const zero_adamw_hparams& h, int64_t t);

// AdamW + cast over n elements of host memory (zero_cpu_adam.cpp).
void cpu_adamw_range(const StepScalars& s, zero_dtype dtype, float* p, float* m, float* v,
                     const float* g, uint16_t* out16, int64_t n);

// Address of the device error word on the current device (nullptr on
// failure), and read-and-clear of it (zero_launch.cu).
int* device_error_word();
int take_device_error(void* stream);

// Launch the bounded-wait self-test kernel (zero_launch.cu).
int launch_selftest_wait(int64_t limit_ns, void* stream);

// Host launchers of the mixed-precision helpers (zero_launch.cu).
int launch_amp_finalize(const NormPartial* partials, int64_t n_tiles, zero_amp_state* state,
                        AmpHead* head, const AmpParams& p, void* stream);
int launch_amp_init(zero_amp_state* state, const zero_amp_state& init, void* stream);

// Host launcher entry (zero_kernels_*.cu): launches `kind` for the jobs in
// `a` on `stream`; returns a CUDA error code (0 on success).
int launch_kernel(Kind kind, zero_dtype dtype, const LaunchArgs& a, void* stream);

}  // namespace zero

// The plan: the library's own description of one parameter group.
struct zero_plan {
  int32_t n_ranks = 0;
  int32_t mode = 0;
  int32_t align = 1;
  int64_t phi = 0;      // real elements
  int64_t padded = 0;   // length of the gathered flat buffer
  std::vector<int64_t> numel;
  std::vector<int64_t> tensor_start;  // flat index of each tensor's first element
  std::vector<int64_t> shard_len;     // per rank
  std::vector<int64_t> shard_flat;    // per rank: flat index of the shard (flat mode) or -1
  struct Seg {
    int64_t tensor, tensor_off, flat_off, shard_off, len;
  };
  std::vector<std::vector<Seg>> segs;  // per rank, increasing flat order
  struct Run {
    int64_t flat_off, shard_off, len;
  };
  std::vector<std::vector<Run>> runs;  // per rank: maximal runs contiguous in both spaces
};
