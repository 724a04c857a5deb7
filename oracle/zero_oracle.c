/*
 * zero_oracle.c -- plain, slow, single-threaded CPU statement of the ZeRO
 * sharded mixed-precision optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library: every definition below is written out again from the pages.
 *
 * Build: cc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (see
 * oracle/__init__.py).  -ffp-contract=off matters: every float operation
 * below must round once to binary32, never fused into an FMA.
 *
 * Sources (page title, section):
 *  [ZeRO-2 blog]  "DeepSpeed ZeRO-2 ... DeepSpeedZeroOptimizer" (discosf.com),
 *                 sections 2.1, 2.2, 4.1-4.4: the group is flattened into one
 *                 contiguous buffer, split into N near-equal partitions (rank
 *                 r owns partition r), the fp32 master is a copy of the
 *                 16-bit partition, a reduce-scatter leaves each rank the
 *                 averaged gradient of its partition, each rank updates only
 *                 its partition, and an all-gather restores the full params.
 *  [cookllm ZeRO] "ZeRO 优化器" (cookllm.com), "参数分配策略": tensor i of
 *                 named_parameters() is owned by rank i % world_size, and an
 *                 AdamW optimizer is built over the owned tensors only;
 *                 "梯度同步": the owner receives the SUM of all ranks'
 *                 gradients (dist.reduce); memory tables for stages 1-3.
 *  [ZeRO report]  "ZeRO / DeepSpeed 深度解读报告" (zako-mio.github.io), §3.3:
 *                 per-device memory 16P, 4P+12P/N, 2P+14P/N, 16P/N.
 *  [wmrh tutorial] "ZeRO ... 实操" (wmrh.cn), §3.1: the AdamW hyper-parameter
 *                 set (lr, betas, eps, weight_decay).
 *
 * Readings where the pages are silent (each one also listed in the design
 * notes):
 *  - "near-equal partition": P = ceil(phi / (N*A)) * N*A, S = P / N, tensors
 *    concatenated with no padding between them, zero padding at the tail only.
 *  - AdamW: the pages name torch.optim.AdamW but print no formula; the
 *    decoupled-decay, bias-corrected form of that class is used, one binary32
 *    rounding per operation, in this order:
 *        p   = p * d                 d  = 1 - lr*wd
 *        m   = b1*m + c1*g           c1 = 1 - b1
 *        v   = b2*v + c2*(g*g)       c2 = 1 - b2
 *        den = sqrt(v)/sb + eps      sb = sqrt(1 - b2^t)
 *        p   = p - ss*(m/den)        ss = lr / (1 - b1^t)
 *    The scalars are formed in binary64 from the caller's values and
 *    rounded once to binary32.
 *  - the reduction accumulates in binary32 in rank order q = 0..N-1 and, for
 *    the average, divides the sum by N once.
 *  - 16-bit rounding is round-to-nearest-even with gradual underflow and
 *    overflow to infinity; a NaN input gives the canonical quiet NaN of the
 *    target format with the input's sign.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_FP16 0
#define ORC_BF16 1
#define ORC_FLAT 0
#define ORC_RR 1
#define ORC_SUM 0
#define ORC_AVG 1

typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} orc_hparams;

/* ------------------------------------------------------------------ */
/* 16-bit formats, from the IEEE 754 binary16 and bfloat16 definitions */
/* ------------------------------------------------------------------ */

static uint32_t bits_of(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float float_of(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/*
 * A finite 16-bit format with `man` stored mantissa bits, exponent bias
 * `bias` and an `expw`-bit exponent field.  Value of a normal number:
 * (2^man + mantissa) * 2^(e - bias - man); of a subnormal:
 * mantissa * 2^(1 - bias - man).
 */
static float decode16(uint16_t h, int man, int expw, int bias) {
  int sign = (h >> 15) & 1;
  int e = (h >> man) & ((1 << expw) - 1);
  int mant = h & ((1 << man) - 1);
  double val;
  if (e == (1 << expw) - 1) {
    if (mant == 0) return sign ? -INFINITY : INFINITY;
    /* NaN: keep sign and payload, made quiet */
    uint32_t u = ((uint32_t)sign << 31) | 0x7f800000u | 0x00400000u |
                 ((uint32_t)mant << (23 - man));
    return float_of(u);
  }
  if (e == 0)
    val = ldexp((double)mant, 1 - bias - man);
  else
    val = ldexp((double)((1 << man) + mant), e - bias - man);
  return (float)(sign ? -val : val); /* exact: every 16-bit value fits in binary32 */
}

/*
 * Round a binary32 value to the nearest value of the 16-bit format, ties to
 * even.  Work on the exact value x = M * 2^E (M integer).  The spacing of the
 * format around |x| is 2^q with q = max(floor(log2|x|) - man, qmin), where
 * qmin is the exponent of the smallest subnormal.  Round |x| / 2^q to an
 * integer k, then encode k * 2^q.
 */
static uint16_t encode16(float x, int man, int expw, int bias) {
  uint32_t u = bits_of(x);
  uint16_t sign = (uint16_t)((u >> 31) << 15);
  int e8 = (u >> 23) & 0xff;
  uint32_t m23 = u & 0x7fffff;
  int emax = (1 << expw) - 1;                  /* all-ones exponent field */
  uint16_t inf = (uint16_t)(sign | (emax << man));
  if (e8 == 0xff) {
    if (m23 == 0) return inf;
    return (uint16_t)(inf | (1 << (man - 1))); /* canonical quiet NaN */
  }
  if (e8 == 0 && m23 == 0) return sign;        /* +-0 */
  uint64_t M;
  int E;
  if (e8 == 0) {
    M = m23;
    E = -149;
  } else {
    M = m23 | 0x800000u;
    E = e8 - 150;
  }
  int lg = 63 - __builtin_clzll(M) + E;        /* floor(log2 |x|), M != 0 */
  int qmin = 1 - bias - man;
  int q = lg - man;
  if (q < qmin) q = qmin;
  int shift = q - E;
  uint64_t k;
  if (shift <= 0) {
    k = M << (-shift);                         /* exactly representable */
  } else if (shift >= 40) {
    k = 0;                                     /* far below half a spacing */
  } else {
    k = M >> shift;
    uint64_t rem = M & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (k & 1))) k++;
  }
  if (k == (2ull << man)) { /* rounding carried into the next binade */
    k >>= 1;
    q++;
  }
  if (k == 0) return sign;
  if (k < (1ull << man)) return (uint16_t)(sign | k); /* subnormal */
  int efield = q + bias + man;
  if (efield >= emax) return inf;               /* overflow */
  return (uint16_t)(sign | (efield << man) | (k - (1ull << man)));
}

uint16_t orc_f32_to_f16(float x) { return encode16(x, 10, 5, 15); }
uint16_t orc_f32_to_bf16(float x) { return encode16(x, 7, 8, 127); }
float orc_f16_to_f32(uint16_t h) { return decode16(h, 10, 5, 15); }
float orc_bf16_to_f32(uint16_t h) { return decode16(h, 7, 8, 127); }

static float to_f32(int dtype, uint16_t h) {
  return dtype == ORC_BF16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

static uint16_t to_16(int dtype, float x) {
  return dtype == ORC_BF16 ? orc_f32_to_bf16(x) : orc_f32_to_f16(x);
}

void orc_f32_to_16_array(int32_t dtype, const uint32_t* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = to_16(dtype, float_of(in[i]));
}

void orc_16_to_f32_array(int32_t dtype, const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = to_f32(dtype, in[i]);
}

/* ------------------------------------------------------------------ */
/* Partition plan                                                      */
/* ------------------------------------------------------------------ */

/*
 * [ZeRO-2 blog] §4.1: flatten the group, split it into N near-equal
 * partitions.  Reading: equal partitions of S = P/N elements with P the
 * element count rounded up to a multiple of N*A.
 */
int orc_plan_flat(const int64_t* numel, int32_t n, int32_t N, int32_t A,
                  int64_t* phi, int64_t* P, int64_t* S) {
  if (n < 0 || N < 1 || A < 1) return 1;
  int64_t total = 0;
  for (int32_t k = 0; k < n; k++) {
    if (numel[k] < 0) return 1;
    total += numel[k];
  }
  int64_t unit = (int64_t)N * A;
  int64_t padded = ((total + unit - 1) / unit) * unit;
  *phi = total;
  *P = padded;
  *S = padded / N;
  return 0;
}

/*
 * The elements rank `rank` owns, as segments (tensor k, offset inside k,
 * flat index, shard index, length), in increasing flat order.
 * Flat mode: every non-empty intersection of tensor k's flat range with
 * [rank*S, (rank+1)*S); the tail padding belongs to no tensor and is reported
 * with tensor index -1.
 * Round-robin mode ([cookllm ZeRO] 参数分配策略): the whole of every tensor k
 * with k % N == rank, in increasing k, packed one after another in the shard.
 */
int orc_segments(const int64_t* numel, int32_t n, int32_t N, int32_t mode, int32_t A,
                 int32_t rank, int64_t* t_idx, int64_t* t_off, int64_t* f_off,
                 int64_t* s_off, int64_t* len, int64_t cap, int64_t* n_out) {
  if (rank < 0 || rank >= N) return 1;
  int64_t count = 0;
#define ORC_EMIT(k_, to_, fo_, so_, l_)          \
  do {                                           \
    if (count < cap) {                           \
      t_idx[count] = (k_);                       \
      t_off[count] = (to_);                      \
      f_off[count] = (fo_);                      \
      s_off[count] = (so_);                      \
      len[count] = (l_);                         \
    }                                            \
    count++;                                     \
  } while (0)
  if (mode == ORC_FLAT) {
    int64_t phi, P, S;
    if (orc_plan_flat(numel, n, N, A, &phi, &P, &S)) return 1;
    int64_t lo = (int64_t)rank * S, hi = lo + S;
    int64_t start = 0; /* flat index of tensor k's first element */
    for (int32_t k = 0; k < n; k++) {
      int64_t end = start + numel[k];
      int64_t a = start > lo ? start : lo;
      int64_t b = end < hi ? end : hi;
      if (a < b) ORC_EMIT(k, a - start, a, a - lo, b - a);
      start = end;
    }
    if (phi < hi) {
      int64_t a = phi > lo ? phi : lo;
      ORC_EMIT(-1, 0, a, a - lo, hi - a);
    }
  } else if (mode == ORC_RR) {
    int64_t start = 0, shard = 0;
    for (int32_t k = 0; k < n; k++) {
      if (numel[k] < 0) return 1;
      if (k % N == rank) {
        if (numel[k] > 0) ORC_EMIT(k, 0, start, shard, numel[k]);
        shard += numel[k];
      }
      start += numel[k];
    }
  } else {
    return 1;
  }
#undef ORC_EMIT
  *n_out = count;
  return 0;
}

/* ------------------------------------------------------------------ */
/* Memory model: [ZeRO report] §3.3, [cookllm ZeRO] stage tables         */
/* ------------------------------------------------------------------ */

static int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

/*
 * Bytes per rank for params (2), grads (2) and fp32 optimizer state (12)
 * per element, as the exact fraction num/den:
 *   stage 0 (DDP): 2 + 2 + 12 everywhere        -> 16 phi
 *   stage 1: optimizer state sharded            -> 4 phi + 12 phi / N
 *   stage 2: gradients sharded as well          -> 2 phi + 14 phi / N
 *   stage 3: parameters sharded as well         -> 16 phi / N
 */
int orc_memory_bytes(int32_t stage, int64_t phi, int32_t N, int64_t* num, int64_t* den) {
  if (N < 1 || phi < 0) return 1;
  int64_t replicated, sharded; /* bytes per element kept whole / split N ways */
  switch (stage) {
    case 0: replicated = 2 + 2 + 12; sharded = 0; break;
    case 1: replicated = 2 + 2; sharded = 12; break;
    case 2: replicated = 2; sharded = 2 + 12; break;
    case 3: replicated = 0; sharded = 2 + 2 + 12; break;
    default: return 1;
  }
  int64_t a = replicated * phi * N + sharded * phi;
  int64_t b = N;
  int64_t g = gcd64(a, b);
  if (g == 0) g = 1;
  *num = a / g;
  *den = b / g;
  return 0;
}

/* ------------------------------------------------------------------ */
/* The per-element step                                                */
/* ------------------------------------------------------------------ */

typedef struct {
  float d, b1, b2, c1, c2, ss, sb, eps;
} orc_scalars;

static orc_scalars make_scalars(const orc_hparams* h, int64_t t) {
  orc_scalars s;
  s.d = (float)(1.0 - h->lr * h->weight_decay);
  s.b1 = (float)h->beta1;
  s.b2 = (float)h->beta2;
  s.c1 = (float)(1.0 - h->beta1);
  s.c2 = (float)(1.0 - h->beta2);
  s.ss = (float)(h->lr / (1.0 - pow(h->beta1, (double)t)));
  s.sb = (float)sqrt(1.0 - pow(h->beta2, (double)t));
  s.eps = (float)h->eps;
  return s;
}

void orc_step_scalars(const orc_hparams* h, int64_t t, float* out8) {
  orc_scalars s = make_scalars(h, t);
  out8[0] = s.d;
  out8[1] = s.b1;
  out8[2] = s.b2;
  out8[3] = s.c1;
  out8[4] = s.c2;
  out8[5] = s.ss;
  out8[6] = s.sb;
  out8[7] = s.eps;
}

/* reduce-scatter of one element: binary32 sum in rank order, /N for the average */
static float reduce_one(int32_t N, int32_t dtype, int32_t op, const uint16_t* g16, int64_t stride) {
  float acc = to_f32(dtype, g16[0]);
  for (int32_t q = 1; q < N; q++) acc = acc + to_f32(dtype, g16[(int64_t)q * stride]);
  if (op == ORC_AVG) acc = acc / (float)N;
  return acc;
}

/* AdamW on one element of a shard; every operation rounds to binary32 */
static void adamw_one(const orc_scalars* s, float g, float* p, float* m, float* v) {
  float pp = *p * s->d;
  float mm = s->b1 * *m + s->c1 * g;
  float gg = g * g;
  float vv = s->b2 * *v + s->c2 * gg;
  float den = sqrtf(vv) / s->sb + s->eps;
  float upd = mm / den;
  pp = pp - s->ss * upd;
  *p = pp;
  *m = mm;
  *v = vv;
}

/* Reduce only, over n elements; grads laid out rank-major (N rows of n). */
void orc_reduce_elements(int64_t n, int32_t N, int32_t dtype, int32_t op,
                         const uint16_t* grads, float* out) {
  for (int64_t i = 0; i < n; i++) out[i] = reduce_one(N, dtype, op, grads + i, n);
}

/* AdamW + cast only, over n elements with binary32 gradients. */
void orc_adamw_elements(int64_t n, int32_t dtype, const float* g, float* master, float* m,
                        float* v, uint16_t* out16, const orc_hparams* h, int64_t t) {
  orc_scalars s = make_scalars(h, t);
  for (int64_t i = 0; i < n; i++) {
    adamw_one(&s, g[i], &master[i], &m[i], &v[i]);
    if (out16) out16[i] = to_16(dtype, master[i]);
  }
}

/* The whole element step (reduce, AdamW, cast) over n gathered elements. */
void orc_update_elements(int64_t n, int32_t N, int32_t dtype, int32_t op,
                         const uint16_t* grads, float* master, float* m, float* v,
                         uint16_t* out16, const orc_hparams* h, int64_t t) {
  orc_scalars s = make_scalars(h, t);
  for (int64_t i = 0; i < n; i++) {
    float g = reduce_one(N, dtype, op, grads + i, n);
    adamw_one(&s, g, &master[i], &m[i], &v[i]);
    if (out16) out16[i] = to_16(dtype, master[i]);
  }
}

/* ------------------------------------------------------------------ */
/* The step over a whole plan                                          */
/* ------------------------------------------------------------------ */

static int for_each_segment(const int64_t* numel, int32_t n, int32_t N, int32_t mode,
                            int32_t A, int32_t rank, int64_t** seg, int64_t* nseg) {
  int64_t cnt = 0;
  int64_t dummy;
  if (orc_segments(numel, n, N, mode, A, rank, &dummy, &dummy, &dummy, &dummy, &dummy, 0, &cnt))
    return 1;
  int64_t* buf = (int64_t*)malloc(sizeof(int64_t) * 5 * (size_t)(cnt ? cnt : 1));
  if (!buf) return 1;
  int64_t got = 0;
  orc_segments(numel, n, N, mode, A, rank, buf, buf + cnt, buf + 2 * cnt, buf + 3 * cnt,
               buf + 4 * cnt, cnt, &got);
  *seg = buf;
  *nseg = cnt;
  return 0;
}

/*
 * One optimizer step for every rank in rank_mask.  grads[q] is rank q's full
 * flat gradient replica (16-bit); master/m/v[r] are rank r's binary32 shard
 * buffers; full16 (nullable) is the gathered flat 16-bit parameter buffer;
 * shard16 (nullable, or with null entries) receives rank r's 16-bit shard.
 * Returns 0, or 1 on a malformed plan.
 */
int orc_step(const int64_t* numel, int32_t n_tensors, int32_t N, int32_t mode, int32_t A,
             int32_t dtype, int32_t op, const uint16_t* const* grads, float* const* master,
             float* const* m, float* const* v, uint16_t* full16, uint16_t* const* shard16,
             const orc_hparams* h, int64_t t, uint64_t rank_mask) {
  orc_scalars s = make_scalars(h, t);
  for (int32_t r = 0; r < N; r++) {
    if (!((rank_mask >> r) & 1)) continue;
    int64_t* seg;
    int64_t nseg;
    if (for_each_segment(numel, n_tensors, N, mode, A, r, &seg, &nseg)) return 1;
    int64_t* flat = seg + 2 * nseg;
    int64_t* shard = seg + 3 * nseg;
    int64_t* len = seg + 4 * nseg;
    for (int64_t j = 0; j < nseg; j++) {
      for (int64_t e = 0; e < len[j]; e++) {
        int64_t f = flat[j] + e, i = shard[j] + e;
        float acc = to_f32(dtype, grads[0][f]);
        for (int32_t q = 1; q < N; q++) acc = acc + to_f32(dtype, grads[q][f]);
        if (op == ORC_AVG) acc = acc / (float)N;
        adamw_one(&s, acc, &master[r][i], &m[r][i], &v[r][i]);
        uint16_t p16 = to_16(dtype, master[r][i]);
        if (full16) full16[f] = p16;
        if (shard16 && shard16[r]) shard16[r][i] = p16;
      }
    }
    free(seg);
  }
  return 0;
}

/* Reduce-scatter alone: out[r][i] = reduced gradient of rank r's element i. */
int orc_reduce_scatter(const int64_t* numel, int32_t n_tensors, int32_t N, int32_t mode,
                       int32_t A, int32_t dtype, int32_t op, const uint16_t* const* grads,
                       float* const* out, uint64_t rank_mask) {
  for (int32_t r = 0; r < N; r++) {
    if (!((rank_mask >> r) & 1)) continue;
    int64_t* seg;
    int64_t nseg;
    if (for_each_segment(numel, n_tensors, N, mode, A, r, &seg, &nseg)) return 1;
    for (int64_t j = 0; j < nseg; j++)
      for (int64_t e = 0; e < seg[4 * nseg + j]; e++) {
        int64_t f = seg[2 * nseg + j] + e, i = seg[3 * nseg + j] + e;
        float acc = to_f32(dtype, grads[0][f]);
        for (int32_t q = 1; q < N; q++) acc = acc + to_f32(dtype, grads[q][f]);
        if (op == ORC_AVG) acc = acc / (float)N;
        out[r][i] = acc;
      }
    free(seg);
  }
  return 0;
}

/* All-gather alone: full16[flat] = shard16[r][shard] over rank r's segments. */
int orc_allgather(const int64_t* numel, int32_t n_tensors, int32_t N, int32_t mode, int32_t A,
                  const uint16_t* const* shard16, uint16_t* full16, uint64_t rank_mask) {
  for (int32_t r = 0; r < N; r++) {
    if (!((rank_mask >> r) & 1)) continue;
    int64_t* seg;
    int64_t nseg;
    if (for_each_segment(numel, n_tensors, N, mode, A, r, &seg, &nseg)) return 1;
    for (int64_t j = 0; j < nseg; j++)
      for (int64_t e = 0; e < seg[4 * nseg + j]; e++)
        full16[seg[2 * nseg + j] + e] = shard16[r][seg[3 * nseg + j] + e];
    free(seg);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Mixed-precision controls: dynamic loss scaling with overflow skip,  */
/* global-norm gradient clipping                                       */
/* ------------------------------------------------------------------ */
/*
 * The pages give these only as configuration ("ZeRO ... 实操" (wmrh.cn)
 * §3.1 and §3.3 ds_config: fp16 loss_scale 0 = dynamic, loss_scale_window
 * 1000, hysteresis 2, min_loss_scale 1; gradient_clipping).  Reading taken:
 *  - the gradients carry the loss scale S; the reduced gradient g (sum or
 *    average of the replicas, as in the plain step) is checked for
 *    non-finite values through its squared norm  sumsq = sum g^2.  Each
 *    square is the binary32 product g*g: the setup the pages configure is
 *    fp16 training with binary32 gradients and master weights (ds_config
 *    fp16 block with amp opt_level O2, "ZeRO ... 实操" §3.3; the fp32
 *    optimizer partition, "DeepSpeed ZeRO-2 ..." §2.1), where the gradient
 *    and every operation on it are binary32 -- the same rule the update
 *    below follows, whose second moment forms this very product.  The
 *    squares are added in binary64, so that (up to binary64 rounding, far
 *    below the rounding of one binary32 square) the sum does not depend on
 *    how the elements are partitioned over ranks or ordered: partitioning
 *    must leave the result unchanged ("ZeRO ... 实操" §2.1, partitioning
 *    changes no dtype or shape).  So sumsq is non-finite exactly when some
 *    g is non-finite or |g| >= 2^64 (its binary32 square overflows);
 *  - non-finite sumsq: the update is skipped (no state, parameter or step
 *    count changes); if more than one overflow is still tolerated the
 *    tolerance drops by one, else S halves (not below min_scale); the
 *    run of good steps restarts;
 *  - finite: norm = sqrt(sumsq)/S is the unscaled global norm; with
 *    max_norm > 0 the clip factor is min(1, max_norm / (norm + 1e-6))
 *    (as torch.nn.utils.clip_grad_norm_), else 1; the gradient multiplier
 *    coef = clip / S is rounded once to binary32 and every element uses
 *    g * coef (one rounding) in the AdamW update of step t = steps + 1;
 *    after `window` consecutive good steps S doubles and the overflow
 *    tolerance is restored.
 */
typedef struct {
  double init_scale, min_scale;
  int32_t window, hysteresis;
  double max_norm;
} orc_amp_config;

typedef struct {
  double scale, norm;
  int64_t step, skipped;
  int32_t good_steps, hysteresis_left, overflow;
  float coef;
} orc_amp_state;

void orc_amp_init(const orc_amp_config* c, orc_amp_state* s) {
  s->scale = c->init_scale;
  s->norm = 0.0;
  s->step = 0;
  s->skipped = 0;
  s->good_steps = 0;
  s->hysteresis_left = c->hysteresis;
  s->overflow = 0;
  s->coef = 1.0f;
}

int orc_step_amp(const int64_t* numel, int32_t n_tensors, int32_t N, int32_t mode, int32_t A,
                 int32_t dtype, int32_t op, const uint16_t* const* grads, float* const* master,
                 float* const* m, float* const* v, uint16_t* full16, uint16_t* const* shard16,
                 const orc_hparams* h, const orc_amp_config* c, orc_amp_state* st,
                 uint64_t rank_mask) {
  float* gbuf[64] = {0};
  int64_t* segs[64] = {0};
  int64_t nsegs[64] = {0};
  double sumsq = 0.0;
  int rc = 0;
  if (N > 64) return 1;
  /* 1. reduce every owned element and accumulate the squared norm */
  for (int32_t r = 0; r < N && !rc; r++) {
    if (!((rank_mask >> r) & 1)) continue;
    if (for_each_segment(numel, n_tensors, N, mode, A, r, &segs[r], &nsegs[r])) {
      rc = 1;
      break;
    }
    int64_t total = 0;
    for (int64_t j = 0; j < nsegs[r]; j++) total += segs[r][4 * nsegs[r] + j];
    gbuf[r] = (float*)malloc(sizeof(float) * (size_t)(total ? total : 1));
    if (!gbuf[r]) {
      rc = 1;
      break;
    }
    for (int64_t j = 0; j < nsegs[r]; j++)
      for (int64_t e = 0; e < segs[r][4 * nsegs[r] + j]; e++) {
        int64_t f = segs[r][2 * nsegs[r] + j] + e, i = segs[r][3 * nsegs[r] + j] + e;
        float acc = to_f32(dtype, grads[0][f]);
        for (int32_t q = 1; q < N; q++) acc = acc + to_f32(dtype, grads[q][f]);
        if (op == ORC_AVG) acc = acc / (float)N;
        gbuf[r][i] = acc;
        float sq = acc * acc; /* the square is a binary32 number, summed in binary64 */
        sumsq += (double)sq;
      }
  }
  if (!rc) {
    /* 2. the loss-scale decision */
    double S = st->scale;
    if (!isfinite(sumsq)) {
      st->overflow = 1;
      st->skipped += 1;
      st->good_steps = 0;
      st->norm = sqrt(sumsq) / S;
      st->coef = 0.0f;
      if (st->hysteresis_left > 1) {
        st->hysteresis_left -= 1;
      } else {
        double half = S / 2.0;
        st->scale = half > c->min_scale ? half : c->min_scale;
      }
    } else {
      double norm = sqrt(sumsq) / S;
      double clip = 1.0;
      if (c->max_norm > 0.0) {
        double q = c->max_norm / (norm + 1e-6);
        if (q < 1.0) clip = q;
      }
      float coef = (float)(clip / S);
      int64_t t = st->step + 1;
      orc_scalars s = make_scalars(h, t);
      /* 3. the update with the scaled and clipped gradient */
      for (int32_t r = 0; r < N; r++) {
        if (!((rank_mask >> r) & 1)) continue;
        for (int64_t j = 0; j < nsegs[r]; j++)
          for (int64_t e = 0; e < segs[r][4 * nsegs[r] + j]; e++) {
            int64_t f = segs[r][2 * nsegs[r] + j] + e, i = segs[r][3 * nsegs[r] + j] + e;
            float g = gbuf[r][i] * coef;
            adamw_one(&s, g, &master[r][i], &m[r][i], &v[r][i]);
            uint16_t p16 = to_16(dtype, master[r][i]);
            if (full16) full16[f] = p16;
            if (shard16 && shard16[r]) shard16[r][i] = p16;
          }
      }
      st->overflow = 0;
      st->norm = norm;
      st->coef = coef;
      st->step = t;
      st->good_steps += 1;
      if (c->window > 0 && st->good_steps >= c->window) {
        st->scale = S * 2.0;
        st->good_steps = 0;
        st->hysteresis_left = c->hysteresis;
      }
    }
  }
  for (int32_t r = 0; r < N; r++) {
    free(gbuf[r]);
    free(segs[r]);
  }
  return rc;
}
