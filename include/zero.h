/*
 * zero.h -- C ABI of the GB300 ZeRO sharded mixed-precision optimizer step.
 *
 * One process, one GPU, N *virtual* data-parallel ranks: rank q's gradient
 * replica and rank r's optimizer shard are separate caller-owned buffers in
 * the same HBM.  The library owns only the partition plan (host memory).
 * Every tensor argument is caller-owned memory the GPU can address: device
 * memory (for example a torch tensor's data_ptr()), or host memory mapped
 * into the GPU's address space at the same address (pinned with
 * cudaHostAlloc / cudaHostRegister under unified addressing).  Host buffers
 * are read and written by the kernels across the host link (NVLink-C2C on
 * Grace-Blackwell), which replaces an explicit copy; they run at the link's
 * bandwidth instead of HBM's.  Every stream argument is a cudaStream_t passed
 * as void* (NULL = the legacy default stream).  Compute calls are
 * asynchronous on that stream, except the three that run the optimizer on
 * host threads (zero_cpu_adamw_shard_step, zero_offload_step,
 * zero_offload_step_amp), which return when the host work is done.
 *
 * Sources (page title, section) for what each call computes:
 *  [ZeRO-2 blog]   "DeepSpeed ZeRO-2 ... DeepSpeedZeroOptimizer" (discosf.com):
 *                  §2.1 and §4.1 flatten + near-equal partition + fp32 master
 *                  cloned from the 16-bit partition; §2.2 and §4.2 bucketed
 *                  reduce-scatter leaving each rank the averaged gradient of
 *                  its partition; §4.3 local update of the rank's partition;
 *                  §4.4 all-gather of the updated partitions.
 *  [cookllm ZeRO]  "ZeRO 优化器" (cookllm.com): 参数分配策略 (tensor i owned
 *                  by rank i % world_size), 梯度同步 (reduce = sum to the
 *                  owner), the per-stage memory tables.
 *  [ZeRO report]   "ZeRO / DeepSpeed 深度解读报告" (zako-mio.github.io) §3.3:
 *                  per-device memory 16P, 4P+12P/N, 2P+14P/N, 16P/N.
 *  [wmrh tutorial] "ZeRO ... 实操" (wmrh.cn) §3.1: AdamW hyper-parameters.
 *
 * Conventions common to every call:
 *  - Every call returns a zero_status and never throws or aborts.  On
 *    failure, zero_last_error() returns a message (thread-local storage,
 *    valid until the next call on the same thread).
 *  - All arguments are validated before anything is launched; a call that
 *    fails validation launches nothing and leaves every output untouched.
 *  - Device pointers must be 16-byte aligned (ZERO_ERR_ALIGN otherwise);
 *    torch allocations are 256-byte aligned.
 *  - Asynchronous device errors surface as ZERO_ERR_CUDA from the next call
 *    or from zero_sync().
 *  - At most 64 virtual ranks; rank_mask bit r selects rank r.  Pointer
 *    arrays are indexed by rank and have n_ranks entries; entries of ranks
 *    outside rank_mask, or whose shard is empty, are not read and may be
 *    NULL.  Likewise any buffer of zero length (a group whose tensors are
 *    all empty has an empty flat buffer) may be NULL.
 *  - Flat indices f run over the gathered flat buffer (length `padded` from
 *    zero_plan_total); shard indices i run over rank r's shard buffers
 *    (length from zero_plan_shard).
 *  - A call may make several launches (one per bucket, and more when a
 *    bucket holds more runs than one launch carries).  Launches of one call
 *    that touch disjoint elements may run concurrently on the GPU; all of
 *    them complete, with their writes visible, before work enqueued on the
 *    stream after the call starts, so stream order between calls holds as
 *    for single kernels (also inside captured CUDA graphs).
 */
#ifndef ZERO_GB300_H_
#define ZERO_GB300_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZERO_OK = 0,
  ZERO_ERR_INVALID = 1,     /* bad argument: null, out of range, size mismatch   */
  ZERO_ERR_ALIGN = 2,       /* a device pointer is not 16-byte aligned           */
  ZERO_ERR_CUDA = 3,        /* CUDA runtime error (launch or asynchronous)       */
  ZERO_ERR_OOM = 4,         /* host allocation failed                            */
  ZERO_ERR_TIMEOUT = 5,     /* a bounded wait on the device gave up (zero_sync)   */
  ZERO_ERR_UNSUPPORTED = 6  /* valid request this build does not implement       */
} zero_status;

typedef enum { ZERO_FP16 = 0, ZERO_BF16 = 1 } zero_dtype;
typedef enum { ZERO_PART_FLAT = 0, ZERO_PART_ROUND_ROBIN = 1 } zero_part_mode;
typedef enum { ZERO_REDUCE_SUM = 0, ZERO_REDUCE_AVG = 1 } zero_reduce_op;

/*
 * AdamW hyper-parameters as the caller holds them (binary64).  The library
 * forms the step's binary32 constants in binary64 and rounds each once:
 *   d = 1 - lr*weight_decay, c1 = 1 - beta1, c2 = 1 - beta2,
 *   ss = lr / (1 - beta1^t), sb = sqrt(1 - beta2^t).
 * Requirements: all finite, lr >= 0, weight_decay >= 0, eps > 0,
 * 0 <= beta1 < 1, 0 <= beta2 < 1.
 */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} zero_adamw_hparams;

typedef struct zero_plan zero_plan; /* opaque, host memory, owned by the library */

/* ------------------------------------------------------------------------ */
/* Partition plan (host only; no GPU needed)                                */
/* ------------------------------------------------------------------------ */

/*
 * Build the partition plan of one parameter group.
 *  numel[k], k < n_tensors: element counts of the group's tensors in
 *    named_parameters() order (>= 0; n_tensors >= 1).
 *  ZERO_PART_FLAT ([ZeRO-2 blog] §2.1, §4.1): the tensors are concatenated
 *    with no gap into one flat buffer of phi = sum(numel) elements, padded at
 *    the tail with zeros to P = ceil(phi / (n_ranks*align_elems)) *
 *    n_ranks*align_elems; rank r owns flat range [r*S, (r+1)*S), S = P/n_ranks.
 *    align_elems must be a power of two in [1, 4096].
 *  ZERO_PART_ROUND_ROBIN ([cookllm ZeRO] 参数分配策略): tensor k is owned
 *    whole by rank k % n_ranks; the flat buffer is the unpadded concatenation
 *    (P = phi) and rank r's shard packs its tensors in increasing k.
 *    align_elems is ignored.
 *  n_ranks in [1, 64].  On success *out receives a plan that the caller
 *  releases with zero_plan_destroy.
 */
zero_status zero_plan_partitions(const int64_t* numel, int32_t n_tensors, int32_t n_ranks,
                                 zero_part_mode mode, int32_t align_elems, zero_plan** out);

/* Release a plan (NULL is allowed). */
void zero_plan_destroy(zero_plan* plan);

/* phi = real element count, padded = length of the gathered flat buffer. */
zero_status zero_plan_total(const zero_plan* plan, int64_t* phi, int64_t* padded);

/* Number of virtual ranks and the partition mode of a plan. */
zero_status zero_plan_info(const zero_plan* plan, int32_t* n_ranks, int32_t* mode,
                           int32_t* align_elems, int32_t* n_tensors);

/*
 * Rank r's shard: *len = its element count; *flat_off = the flat index of its
 * first element in flat mode, or -1 in round-robin mode (shards are not
 * contiguous in the flat buffer there).
 */
zero_status zero_plan_shard(const zero_plan* plan, int32_t rank, int64_t* flat_off,
                            int64_t* len);

/*
 * Ownership map of rank r: the segments (tensor_idx, tensor_off, flat_off,
 * shard_off, len) in increasing flat order.  A segment is a maximal run of
 * elements that lies in one tensor and in rank r's shard; flat-mode tail
 * padding is reported with tensor_idx = -1.  Each output array holds `cap`
 * entries; *n_out receives the number of segments (which may exceed cap: call
 * once with cap = 0 to size the arrays).  Output arrays may be NULL when
 * cap == 0.
 */
zero_status zero_plan_segments(const zero_plan* plan, int32_t rank, int64_t* tensor_idx,
                               int64_t* tensor_off, int64_t* flat_off, int64_t* shard_off,
                               int64_t* len, int64_t cap, int64_t* n_out);

/* Human-readable dump of the plan into buf (NUL-terminated, truncated to cap). */
zero_status zero_plan_describe(const zero_plan* plan, char* buf, int64_t cap);

/*
 * Per-rank model-state bytes of mixed-precision Adam training ([ZeRO report]
 * §3.3; [cookllm ZeRO] stage tables): 2 B/param 16-bit params, 2 B/param
 * 16-bit grads, 12 B/param fp32 master + m + v.  stage 0 (DDP) 16 phi;
 * 1: 4 phi + 12 phi/N; 2: 2 phi + 14 phi/N; 3: 16 phi/N.  Returned as the
 * exact reduced fraction *num / *den.  ZERO_ERR_INVALID if the numerator
 * would overflow int64.
 */
zero_status zero_memory_bytes(int32_t stage, int64_t phi, int32_t n_ranks, int64_t* num,
                              int64_t* den);

/* ------------------------------------------------------------------------ */
/* Device calls                                                             */
/* ------------------------------------------------------------------------ */

/*
 * Optimizer-state initialisation ([ZeRO-2 blog] §4.1: each rank clones its
 * fp32 master from its own 16-bit partition):
 *   master[r][i] = float(full_flat16[f]), m[r][i] = v[r][i] = +0
 * for every (f, i) owned by a rank in rank_mask.  The widening is exact.
 *  full_flat16: device, `padded` 16-bit elements of `dtype` (read).
 *  master/m/v:  n_ranks device pointers, each to that rank's shard length of
 *               float (written).
 */
zero_status zero_init_shards(const zero_plan* plan, const void* full_flat16, zero_dtype dtype,
                             float* const* master, float* const* m, float* const* v,
                             uint64_t rank_mask, void* stream);

/*
 * Reduce-scatter ([ZeRO-2 blog] §2.2, §4.2; [cookllm ZeRO] 梯度同步):
 *   grad_shards[r][i] = G_0[f] + G_1[f] + ... + G_{N-1}[f]
 * accumulated in binary32 in rank order, then divided by N for
 * ZERO_REDUCE_AVG.  grads[q] (n_ranks entries, all required) points to rank
 * q's flat gradient replica of `dtype`; it is read only at the flat indices
 * owned by ranks in rank_mask (so a caller holding only those ranges may pass
 * correspondingly offset pointers).  grad_shards[r]: device float[shard len].
 *  bucket_elems > 0 splits the work into buckets of that many flat indices,
 *  one launch each (like the reduce_bucket_size of the pages); <= 0 means one
 *  bucket.  Results do not depend on the bucketing.
 */
zero_status zero_reduce_scatter(const zero_plan* plan, const void* const* grads,
                                zero_dtype dtype, zero_reduce_op op, float* const* grad_shards,
                                uint64_t rank_mask, int64_t bucket_elems, void* stream);

/*
 * zero_reduce_scatter restricted to the flat index range [flat_lo, flat_hi)
 * (0 <= flat_lo <= flat_hi <= padded): one gradient bucket.  This is the call
 * a backward pass makes as soon as every rank's replica holds a bucket's
 * gradients ("DeepSpeed ZeRO-2 ..." §2.2, §4.2: IPG buckets of
 * reduce_bucket_size reduced on a side stream while the backward pass goes
 * on, overlap_comm).  Only grad_shards elements whose flat index falls in the
 * range are written; an empty intersection launches nothing.
 */
zero_status zero_reduce_scatter_range(const zero_plan* plan, const void* const* grads,
                                      zero_dtype dtype, zero_reduce_op op,
                                      float* const* grad_shards, uint64_t rank_mask,
                                      int64_t flat_lo, int64_t flat_hi, void* stream);

/*
 * Local AdamW step on each masked rank's shard ([ZeRO-2 blog] §4.3), one
 * binary32 rounding per operation, in this order (t = step >= 1):
 *   p = p*d;  m = b1*m + c1*g;  v = b2*v + c2*(g*g);
 *   den = sqrt(v)/sb + eps;  p = p - ss*(m/den)
 * and, when out16_shard is non-NULL, out16_shard[r][i] = p rounded to
 * nearest even in `dtype` (entries may be NULL to skip a rank).
 *  master/m/v: device float[shard len] (read-modify-write).
 *  grad_shards: device float[shard len] (read).
 */
zero_status zero_adamw_shard_step(const zero_plan* plan, float* const* master, float* const* m,
                                  float* const* v, const float* const* grad_shards,
                                  void* const* out16_shard, zero_dtype dtype,
                                  const zero_adamw_hparams* hp, int64_t step,
                                  uint64_t rank_mask, void* stream);

/*
 * ZeRO-Offload's CPU optimizer ([ZeRO-2 blog] §4.5: offload_optimizer to the
 * CPU, DeepSpeedCPUAdam, pinned buffers): the update of
 * zero_adamw_shard_step computed by host threads on HOST buffers (master, m,
 * v, grad_shards and out16_shard are host memory, pinned or not), with the
 * same binary32 operations in the same order, so the results equal the GPU
 * update bit for bit.  It runs only when called: the usual offload step is
 * zero_reduce_scatter into pinned host grad_shards, zero_sync, this call,
 * then zero_allgather from the pinned host 16-bit shards (zero_offload_step
 * runs that sequence overlapped).  Synchronous; the masked ranks' shards are
 * split into n_threads equal slices (n_threads <= 0: every hardware thread;
 * the calling thread takes the first slice).
 */
zero_status zero_cpu_adamw_shard_step(const zero_plan* plan, float* const* master,
                                      float* const* m, float* const* v,
                                      const float* const* grad_shards, void* const* out16_shard,
                                      zero_dtype dtype, const zero_adamw_hparams* hp,
                                      int64_t step, uint64_t rank_mask, int32_t n_threads);

/*
 * ZeRO-Offload with the CPU optimizer, pipelined ([ZeRO-2 blog] §4.5:
 * offload_optimizer to the CPU, DeepSpeedCPUAdam, pinned-memory gradient
 * buffers; the pipelining is this library's).  The result is that of
 *   zero_reduce_scatter(grads -> grad_shards); zero_sync;
 *   zero_cpu_adamw_shard_step(master, m, v, grad_shards -> out16_shard);
 *   zero_allgather(out16_shard -> full_flat16)
 * element for element and bit for bit, but the flat index space is cut into
 * chunks of chunk_elems elements: the device reduces every chunk in turn,
 * host threads update chunk k as soon as its reduction has completed (while
 * the device still reduces the chunks after it), and chunk k's all-gather is
 * enqueued as soon as the host has written its 16-bit values.
 *  grads: the N flat replicas (device, or pinned host memory); or NULL when
 *    grad_shards already hold the reduced gradients (reduced bucket by bucket
 *    during backward): then nothing is reduced, `op` is not used, and the
 *    host update starts once the work enqueued on `stream` before the call
 *    has completed (the update and the gathers still overlap).
 *  grad_shards, out16_shard: PINNED (or managed) host memory the device
 *    writes (fp32 reduced gradient) and reads (16-bit shard) across the host
 *    link; checked with cudaPointerGetAttributes (ZERO_ERR_INVALID otherwise).
 *  master, m, v: host memory (pinned or not; never device memory), updated
 *    by the host threads only.
 *  full_flat16: device memory, or NULL for no gather (the 16-bit shards are
 *    still written).
 *  chunk_elems <= 0: one chunk (no overlap); at most 4096 chunks.
 *  n_threads: host threads that update (at most 1024); <= 0: every hardware
 *    thread but one, which is left to the calling thread (it sleeps on the
 *    device's events and launches the gathers).
 * Each thread updates an equal slice of every chunk, so the host part takes
 * what streaming 30 bytes per element through host memory takes; the device
 * traffic across the host link shares that memory.
 * Blocking: returns when every host update is done and every gather is
 * enqueued on `stream` (the gathers complete asynchronously; zero_sync or a
 * later call on `stream` orders after them).  It waits for the device in the
 * middle, so it cannot be captured in a CUDA graph (ZERO_ERR_UNSUPPORTED
 * while `stream` is capturing).  A ZERO_ERR_CUDA during the call may leave
 * some chunks updated and others not.
 */
zero_status zero_offload_step(const zero_plan* plan, const void* const* grads, zero_dtype dtype,
                              zero_reduce_op op, float* const* grad_shards, float* const* master,
                              float* const* m, float* const* v, void* const* out16_shard,
                              void* full_flat16, const zero_adamw_hparams* hp, int64_t step,
                              uint64_t rank_mask, int64_t chunk_elems, int32_t n_threads,
                              void* stream);

/*
 * All-gather ([ZeRO-2 blog] §4.4): full_flat16[f] = shards16[r][i] for every
 * (f, i) owned by a rank in rank_mask.  Flat-mode tail padding belongs to
 * the last rank's shard and is copied like any other element.
 */
zero_status zero_allgather(const zero_plan* plan, const void* const* shards16,
                           zero_dtype dtype, void* full_flat16, uint64_t rank_mask,
                           void* stream);

/*
 * The fused step: reduce-scatter, AdamW, cast and all-gather in one pass
 * over HBM (one read of the N gradient replicas and of master/m/v, one write
 * of master/m/v and of the 16-bit parameters).  The results are bit-identical
 * to zero_reduce_scatter -> zero_adamw_shard_step -> zero_allgather.
 *  full_flat16 (nullable): gathered flat 16-bit buffer, written at the flat
 *    indices of masked ranks.
 *  out16_shard (nullable, entries nullable): each rank's 16-bit shard (the
 *    ZeRO-3 layout, where the shard is the next all-gather's source).
 *  bucket_elems: as for zero_reduce_scatter.
 */
zero_status zero_step(const zero_plan* plan, const void* const* grads, zero_dtype dtype,
                      zero_reduce_op op, float* const* master, float* const* m, float* const* v,
                      void* full_flat16, void* const* out16_shard, const zero_adamw_hparams* hp,
                      int64_t step, uint64_t rank_mask, int64_t bucket_elems, void* stream);

/* ------------------------------------------------------------------------ */
/* ZeRO-3 layer stream with prefetch                                        */
/* ------------------------------------------------------------------------ */
/*
 * ZeRO-3 keeps only 16-bit shards of every layer and gathers a layer's full
 * parameters just before it is used, releasing them afterwards ("ZeRO 优化器"
 * (cookllm.com), ZeRO Stage 3: per-layer gather -> compute -> release;
 * "ZeRO / DeepSpeed 深度解读报告" §2.4; "DeepSpeed ZeRO-2 ..." §5 names the
 * prefetch bucket).  One layer of a stack that shares one plan: */
typedef struct {
  const void* const* grads; /* n_ranks 16-bit flat gradient replicas of the layer   */
  float* const* master;     /* n_ranks fp32 shards (read-modify-write)               */
  float* const* m;          /* n_ranks fp32 shards (read-modify-write)               */
  float* const* v;          /* n_ranks fp32 shards (read-modify-write)               */
  void* const* shards16;    /* n_ranks 16-bit shards: gather source, step output     */
} zero_layer;

/*
 * One pass over n_layers layers: for layer l, zero_allgather(shards16 ->
 * layer_bufs[l % n_bufs]) on gather_stream, then zero_step(grads, master, m,
 * v, full_flat16 = NULL, out16_shard = shards16) on step_stream for step
 * `step`.  Ordering, enforced with events (no host waits):
 *   - the gather of layer l starts after the step of layer l - n_bufs
 *     finished (the layer buffer it overwrites is released then);
 *   - the step of layer l starts after the gather of layer l (the step
 *     rewrites the shards the gather reads);
 *   - the first gather starts after all work already queued on step_stream.
 * So with two streams and n_bufs >= 2 the gathers of the next layers run
 * ahead (prefetch) while earlier layers update; with gather_stream ==
 * step_stream the pass is serial.  All work of the pass is complete once
 * step_stream reaches the point after the call.  Results do not depend on
 * n_bufs or the streams.  n_bufs in [1, 64]; every layer buffer holds
 * `padded` 16-bit elements.
 */
zero_status zero_zero3_pass(const zero_plan* plan, const zero_layer* layers, int32_t n_layers,
                            void* const* layer_bufs, int32_t n_bufs, zero_dtype dtype,
                            zero_reduce_op op, const zero_adamw_hparams* hp, int64_t step,
                            void* gather_stream, void* step_stream);

/* ------------------------------------------------------------------------ */
/* Mixed-precision controls: dynamic loss scaling, overflow skip, clipping  */
/* ------------------------------------------------------------------------ */
/*
 * The pages give these as configuration only ("ZeRO ... 实操" (wmrh.cn) §3.1
 * and §3.3, ds_config: fp16 loss_scale 0 (dynamic), loss_scale_window,
 * hysteresis, min_loss_scale; gradient_clipping).  What the library does:
 *  - the gradient replicas carry the loss scale S; they are reduced as by
 *    zero_reduce_scatter into binary32 shards, and the squared L2 norm of
 *    the reduced gradient over every masked rank is accumulated (binary32
 *    squares; sums in a fixed order with about 48 significant bits, kept as
 *    pairs of binary32 numbers, squares of 2^64 and above in a second pair
 *    scaled by 2^-64, so the sum of finite squares is finite);
 *  - a non-finite norm (an inf or NaN anywhere) skips the update: no
 *    parameter, moment or step count changes; if more than one overflow is
 *    still tolerated the tolerance drops by one, else S halves (not below
 *    min_scale); the run of good steps restarts;
 *  - otherwise norm = sqrt(sumsq)/S; the clip factor is
 *    min(1, max_norm/(norm + 1e-6)) when max_norm > 0 (as
 *    torch.nn.utils.clip_grad_norm_), else 1; every element's gradient is
 *    g * coef with coef = clip/S rounded once to binary32, and AdamW runs as
 *    zero_adamw_shard_step for step t = state.step + 1, followed by the cast
 *    and the all-gather of zero_step; after `window` consecutive good steps S
 *    doubles and the overflow tolerance is restored.
 * Every decision is taken on the device: no call waits for the host, so a
 * sequence of steps needs no synchronisation.
 */
typedef struct {
  double init_scale;  /* loss scale of the first gradients (finite, > 0)           */
  double min_scale;   /* floor of the loss scale (finite, > 0)                       */
  int32_t window;     /* good steps before the scale doubles; 0 = never grows        */
  int32_t hysteresis; /* overflows tolerated before the scale halves (>= 1)          */
  double max_norm;    /* clip threshold of the unscaled global norm; <= 0 = no clip  */
} zero_amp_config;

/* State of the controls; lives in caller-owned DEVICE memory (16-byte aligned),
 * written by zero_amp_init and by every zero_step_amp; copy it to the host to
 * read it. */
typedef struct {
  double scale;            /* loss scale the next gradients are expected to carry */
  double norm;             /* unscaled global L2 norm of the last call (inf/NaN on overflow) */
  int64_t step;            /* AdamW steps applied (skipped calls not counted)     */
  int64_t skipped;         /* calls skipped because of a non-finite gradient      */
  int32_t good_steps;      /* good steps since the scale last changed             */
  int32_t hysteresis_left; /* overflows still tolerated before the scale halves   */
  int32_t overflow;        /* 1 if the last call skipped its update               */
  float coef;              /* gradient multiplier of the last applied update      */
  float sc[8];             /* binary32 AdamW constants of the last applied update */
} zero_amp_state;

/* Write the initial state (scale = init_scale, everything else 0, tolerance =
 * hysteresis) into d_state, asynchronously on `stream`. */
zero_status zero_amp_init(void* d_state, const zero_amp_config* cfg, void* stream);

/* Bytes of device workspace zero_step_amp needs for this plan, mask and
 * bucketing: an 8 KB head (copies of the step's decision record, the
 * decision kernel's partial sums) plus one 16-byte partial sum of squares
 * per 2048-element tile. */
zero_status zero_amp_workspace_bytes(const zero_plan* plan, uint64_t rank_mask,
                                     int64_t bucket_elems, int64_t* bytes);

/*
 * One mixed-precision step (see above).  Arguments as zero_step, plus:
 *  grad_shards: n_ranks device pointers to float[shard len], written with the
 *    reduced (still scaled) gradient, the partitioned gradient of ZeRO-2;
 *  cfg: host pointer, read during the call;
 *  d_state: the device state (read-modify-write);
 *  workspace: caller-owned device scratch of at least
 *    zero_amp_workspace_bytes(plan, rank_mask, bucket_elems), 16-byte aligned.
 * Launches the reduction (one launch per bucket), the decision kernel and
 * the update; calls must not overlap on the device when they share d_state
 * or workspace.
 */
zero_status zero_step_amp(const zero_plan* plan, const void* const* grads, zero_dtype dtype,
                          zero_reduce_op op, float* const* grad_shards, float* const* master,
                          float* const* m, float* const* v, void* full_flat16,
                          void* const* out16_shard, const zero_adamw_hparams* hp,
                          const zero_amp_config* cfg, void* d_state, void* workspace,
                          int64_t workspace_bytes, uint64_t rank_mask, int64_t bucket_elems,
                          void* stream);

/*
 * The mixed-precision step from gradients that are already reduce-scattered:
 * grad_shards[r] (read only) holds rank r's reduced, still loss-scaled fp32
 * gradient, as zero_reduce_scatter or zero_reduce_scatter_range leave it --
 * the flow of a training loop that reduces gradient buckets while the
 * backward pass runs ("DeepSpeed ZeRO-2 ..." §2.2, §4.2: overlap_comm and the
 * reduction stream) and then checks for overflow, clips and updates the
 * partitions.  Everything else (norm, skip, loss scale, clip, AdamW, cast,
 * gather, workspace, state) is as zero_step_amp; the workspace size is
 * zero_amp_workspace_bytes(plan, rank_mask, bucket_elems) for the same
 * bucket_elems.  The results equal zero_reduce_scatter followed by this call
 * and zero_step_amp on the replicas, bit for bit.
 */
zero_status zero_step_amp_shards(const zero_plan* plan, zero_dtype dtype,
                                 float* const* grad_shards, float* const* master, float* const* m,
                                 float* const* v, void* full_flat16, void* const* out16_shard,
                                 const zero_adamw_hparams* hp, const zero_amp_config* cfg,
                                 void* d_state, void* workspace, int64_t workspace_bytes,
                                 uint64_t rank_mask, int64_t bucket_elems, void* stream);

/*
 * One gradient bucket of a mixed-precision training step: the reduce-scatter
 * of zero_reduce_scatter_range over the flat range
 * [bucket_index * bucket_elems, min((bucket_index + 1) * bucket_elems,
 * padded)) (bucket_elems <= 0: one bucket, the whole buffer), which also
 * writes that bucket's per-tile sums of squares into `workspace`, numbered
 * exactly as zero_step_amp numbers its tiles for the same plan, rank_mask
 * and bucket_elems -- the reduction the pages overlap with the backward pass
 * ("DeepSpeed ZeRO-2 ..." §2.2, §4.2: reduce_bucket_size, overlap_comm),
 * with the overflow check's and the clipping norm's first pass folded into
 * it, so that zero_step_amp_reduced needs no pass over the gradient shards
 * for them.  Buckets may be reduced in any order, on any stream ordered
 * before the step.  The launch holding the step's first tile also prepares
 * the decision (it reads d_state's step count: no step on this state may be
 * in flight).
 *  hp: host pointer, read during the call (beta1, beta2);
 *  d_state: the device state of zero_amp_init (read);
 *  workspace: as zero_step_amp's, of at least
 *    zero_amp_workspace_bytes(plan, rank_mask, bucket_elems) bytes.
 * Errors: bucket_index outside the buckets, an undersized workspace, and
 * the argument errors of zero_reduce_scatter_range (ZERO_ERR_INVALID /
 * ZERO_ERR_ALIGN), before any launch.  A bucket whose range holds no element
 * of a masked rank launches nothing.
 */
zero_status zero_reduce_scatter_bucket_amp(const zero_plan* plan, const void* const* grads,
                                           zero_dtype dtype, zero_reduce_op op,
                                           float* const* grad_shards,
                                           const zero_adamw_hparams* hp, const void* d_state,
                                           void* workspace, int64_t workspace_bytes,
                                           uint64_t rank_mask, int64_t bucket_elems,
                                           int64_t bucket_index, void* stream);

/*
 * The mixed-precision step after every bucket of the plan was reduced by
 * zero_reduce_scatter_bucket_amp into grad_shards and `workspace` with the
 * same rank_mask and bucket_elems since the last step on this state: only
 * the decision kernel and the update run (no pass over the gradient shards
 * for the norm: 30 bytes per element instead of zero_step_amp_shards's 34).
 * Arguments and results as zero_step_amp_shards; the results equal
 * zero_step_amp on the replicas with the same bucket_elems, bit for bit.
 * Calling it without those reductions decides on whatever the workspace
 * holds (nothing checks this on the device).
 */
zero_status zero_step_amp_reduced(const zero_plan* plan, zero_dtype dtype,
                                  float* const* grad_shards, float* const* master,
                                  float* const* m, float* const* v, void* full_flat16,
                                  void* const* out16_shard, const zero_adamw_hparams* hp,
                                  const zero_amp_config* cfg, void* d_state, void* workspace,
                                  int64_t workspace_bytes, uint64_t rank_mask,
                                  int64_t bucket_elems, void* stream);

/*
 * The mixed-precision step with the optimizer offloaded to the host
 * ([ZeRO-2 blog] §4.5 with the fp16 controls above): the device reduces
 * (grads non-NULL, as zero_step_amp; or grads NULL, the shards and the
 * workspace's sums of squares written by zero_reduce_scatter_bucket_amp with
 * this bucket_elems, as zero_step_amp_reduced) and takes the decision in
 * d_state; the host reads the decision and, unless it skips the step, host
 * threads apply the update of zero_step_amp (gradient times the decision's
 * coef, then AdamW with its constants) to the host master/m/v and write the
 * host 16-bit shards, chunk by chunk, each chunk's gather into full_flat16
 * (nullable) enqueued as soon as it is written.  Buffers, chunk_elems,
 * n_threads, blocking and capture as zero_offload_step; d_state and
 * workspace are device memory as for zero_step_amp.  A skipped step changes
 * nothing on the host and launches no gather.  Results equal zero_step_amp's
 * bit for bit.
 */
zero_status zero_offload_step_amp(const zero_plan* plan, const void* const* grads,
                                  zero_dtype dtype, zero_reduce_op op, float* const* grad_shards,
                                  float* const* master, float* const* m, float* const* v,
                                  void* const* out16_shard, void* full_flat16,
                                  const zero_adamw_hparams* hp, const zero_amp_config* cfg,
                                  void* d_state, void* workspace, int64_t workspace_bytes,
                                  uint64_t rank_mask, int64_t bucket_elems, int64_t chunk_elems,
                                  int32_t n_threads, void* stream);

/*
 * zero_step_amp without a workspace argument, for callers that cannot
 * allocate device memory: code whose device memory all comes from a fixed
 * budget or pool it does not control, or that runs where a cudaMalloc /
 * cudaFree (and the device-wide synchronisation a cudaFree can imply) is not
 * allowed, or that has nowhere to keep a workspace alive between calls.
 * The pages describe no such call; it is a convenience of this library.
 *
 * Same arguments and results as zero_step_amp, minus workspace and
 * workspace_bytes.  The scratch is instead a fixed 2 MiB array compiled into
 * the library, present on every GPU that loads it until the process exits;
 * this call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine).  Limits and rules:
 *  - the step may span at most 130,560 tiles of 2048 elements, i.e.
 *    zero_amp_workspace_bytes(plan, rank_mask, bucket_elems) <= 2 MiB (about
 *    267 million owned elements per call); larger steps are rejected with
 *    ZERO_ERR_INVALID and a message, and nothing is launched;
 *  - the first call on a device looks up the array's device address with
 *    that device current and caches it; make that first call before any
 *    stream capture begins.  With CUDA's lazy module loading (the default)
 *    that lookup is also what loads the library's device code on that
 *    device and commits the 2 MiB array, so the first call can fail with
 *    ZERO_ERR_CUDA (out of memory) on a device that is already full; later
 *    calls commit nothing;
 *  - the cached address belongs to the device's current context: do not call
 *    cudaDeviceReset on that device between calls of this function;
 *  - every call on a device shares the one array, which keeps what the last
 *    call left there (each call writes everything it reads, so nothing needs
 *    clearing): calls whose work overlaps on the GPU (different streams,
 *    not ordered by events) race on it and must be serialised by the caller.
 */
zero_status zero_step_amp_noalloc(const zero_plan* plan, const void* const* grads,
                                  zero_dtype dtype, zero_reduce_op op, float* const* grad_shards,
                                  float* const* master, float* const* m, float* const* v,
                                  void* full_flat16, void* const* out16_shard,
                                  const zero_adamw_hparams* hp, const zero_amp_config* cfg,
                                  void* d_state, uint64_t rank_mask, int64_t bucket_elems,
                                  void* stream);

/*
 * Measurement helper; the pages have no counterpart.  Launches, on `stream`,
 * kernels with exactly the grid, job table and memory accesses zero_step
 * would use for the same arguments (same plan, mask and buckets), but with
 * none of its arithmetic, so that a benchmark can time the floor a launch of
 * that shape reaches on this GPU:
 *   kind 0  the launches alone (every CTA returns at once);
 *   kind 1  every load of the step (the N gradient replicas, master, m, v),
 *           no store;
 *   kind 2  every load and every store of the step: master/m/v are written
 *           back unchanged and full_flat16 (nullable) receives the master
 *           rounded to 16 bits, which is what a step leaves there anyway.
 * No buffer changes value.  Arguments, layouts, ownership and errors as for
 * zero_step (no hyper-parameters, no shard outputs); kind outside 0..2 is
 * ZERO_ERR_INVALID.  Asynchronous on `stream`.
 */
zero_status zero_floor_probe(const zero_plan* plan, int32_t kind, const void* const* grads,
                             zero_dtype dtype, float* const* master, float* const* m,
                             float* const* v, void* full_flat16, uint64_t rank_mask,
                             int64_t bucket_elems, void* stream);

/* Synchronize `stream` and report any asynchronous device error, and
 * ZERO_ERR_TIMEOUT if a kernel gave up a bounded wait since the last check
 * (the device error word is then cleared). */
zero_status zero_sync(void* stream);

/*
 * Self-test of the timeout path: one kernel waits on a barrier that nothing
 * ever completes, gives up after limit_ns nanoseconds (1e3 .. 1e10) and
 * raises the device error word, so the next zero_sync(stream) returns
 * ZERO_ERR_TIMEOUT.  No fault and no hang: the context stays usable.  The
 * library's only waiting kernels (the optional bulk-copy staging of the
 * fused step) give up the same way, after one second.
 */
zero_status zero_selftest_wait_timeout(int64_t limit_ns, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* zero_last_error(void);

/* Number of kernel launches the library issued since load (all threads). */
int64_t zero_launch_count(void);

/* Library version string. */
const char* zero_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H_ */
