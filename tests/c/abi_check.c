/*
 * A plain-C caller of the library's ABI (include/zero.h): no Python, no
 * torch.  Mode "host" checks the plan, the memory model and argument
 * rejection (no GPU needed); mode "gpu" allocates device buffers with the
 * CUDA runtime, runs zero_init_shards + two zero_step calls on a small
 * group and compares the results with the CPU oracle, which this test links
 * as a separate library (the two share no code); mode "amp" runs the
 * mixed-precision step twice over -- zero_step_amp, and the bucket
 * reductions that write the norm's partial sums followed by
 * zero_step_amp_reduced -- requires the two to agree bit for bit and both
 * to match the oracle's mixed-precision step; mode "offload" runs
 * zero_offload_step with the optimizer state in plain malloc'd host memory
 * and the gradient / 16-bit shards in cudaHostAlloc'd memory, two steps in
 * ragged chunks on 3 host threads, against the oracle.
 *
 * Exit status 0 on success; prints the first mismatch otherwise.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero.h"

/* the oracle's C interface (oracle/zero_oracle.c) */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} orc_hparams;
int orc_plan_flat(const int64_t*, int32_t, int32_t, int32_t, int64_t*, int64_t*, int64_t*);
int orc_step(const int64_t*, int32_t, int32_t, int32_t, int32_t, int32_t, int32_t,
             const uint16_t* const*, float* const*, float* const*, float* const*, uint16_t*,
             uint16_t* const*, const orc_hparams*, int64_t, uint64_t);
uint16_t orc_f32_to_bf16(float);
float orc_bf16_to_f32(uint16_t);
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
void orc_amp_init(const orc_amp_config*, orc_amp_state*);
int orc_step_amp(const int64_t*, int32_t, int32_t, int32_t, int32_t, int32_t, int32_t,
                 const uint16_t* const*, float* const*, float* const*, float* const*, uint16_t*,
                 uint16_t* const*, const orc_hparams*, const orc_amp_config*, orc_amp_state*,
                 uint64_t);

#define CHECK(c, ...)                  \
  do {                                 \
    if (!(c)) {                        \
      fprintf(stderr, __VA_ARGS__);    \
      fprintf(stderr, "\n");           \
      return 1;                        \
    }                                  \
  } while (0)

static const int64_t kNumel[] = {1000, 37, 4096, 3, 129, 8191};
enum { kTensors = 6, kRanks = 4, kAlign = 16 };

static int host_checks(void) {
  zero_plan* plan = NULL;
  CHECK(zero_plan_partitions(kNumel, kTensors, kRanks, ZERO_PART_FLAT, kAlign, &plan) == ZERO_OK,
        "plan: %s", zero_last_error());
  int64_t phi, padded, ophi, oP, oS;
  CHECK(zero_plan_total(plan, &phi, &padded) == ZERO_OK, "total");
  CHECK(orc_plan_flat(kNumel, kTensors, kRanks, kAlign, &ophi, &oP, &oS) == 0, "oracle plan");
  CHECK(phi == ophi && padded == oP, "plan totals %lld/%lld vs oracle %lld/%lld",
        (long long)phi, (long long)padded, (long long)ophi, (long long)oP);
  for (int r = 0; r < kRanks; ++r) {
    int64_t off, len;
    CHECK(zero_plan_shard(plan, r, &off, &len) == ZERO_OK, "shard");
    CHECK(off == r * oS && len == oS, "shard %d: %lld+%lld", r, (long long)off, (long long)len);
  }
  int64_t num, den;
  CHECK(zero_memory_bytes(2, 1000000, 8, &num, &den) == ZERO_OK, "memory");
  CHECK(num == 3750000 && den == 1, "stage 2 bytes %lld/%lld", (long long)num, (long long)den);
  /* a NULL plan and a misaligned pointer are rejected before any launch */
  const int64_t before = zero_launch_count();
  zero_adamw_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  void* ptrs[kRanks] = {(void*)0x100000, (void*)0x100000, (void*)0x100000, (void*)0x100008};
  CHECK(zero_step(NULL, (const void* const*)ptrs, ZERO_BF16, ZERO_REDUCE_AVG, (float* const*)ptrs,
                  (float* const*)ptrs, (float* const*)ptrs, NULL, NULL, &hp, 1, 0xF, 0,
                  NULL) == ZERO_ERR_INVALID, "NULL plan accepted");
  CHECK(zero_step(plan, (const void* const*)ptrs, ZERO_BF16, ZERO_REDUCE_AVG, (float* const*)ptrs,
                  (float* const*)ptrs, (float* const*)ptrs, NULL, NULL, &hp, 1, 0xF, 0,
                  NULL) == ZERO_ERR_ALIGN, "misaligned pointer accepted");
  CHECK(zero_launch_count() == before, "a rejected call launched");
  zero_plan_destroy(plan);
  printf("host ok\n");
  return 0;
}

static uint32_t lcg(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;
  return *s;
}

static int gpu_checks(void) {
  zero_plan* plan = NULL;
  CHECK(zero_plan_partitions(kNumel, kTensors, kRanks, ZERO_PART_FLAT, kAlign, &plan) == ZERO_OK,
        "plan");
  int64_t phi, P, S, off;
  zero_plan_total(plan, &phi, &P);
  zero_plan_shard(plan, 0, &off, &S);
  /* host data: parameters and 2 steps x 4 replicas of bf16 gradients */
  uint16_t* p16 = calloc((size_t)P, 2);
  uint16_t* g16[2][kRanks];
  uint32_t seed = 12345u;
  for (int64_t i = 0; i < phi; ++i)
    p16[i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.05f);
  for (int t = 0; t < 2; ++t)
    for (int q = 0; q < kRanks; ++q) {
      g16[t][q] = calloc((size_t)P, 2);
      for (int64_t i = 0; i < phi; ++i)
        g16[t][q][i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.02f);
    }
  /* device buffers */
  void *d_full, *d_p16, *d_g[kRanks];
  float *d_m[kRanks], *d_v[kRanks], *d_master[kRanks];
  CHECK(cudaMalloc(&d_full, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&d_p16, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(d_p16, p16, (size_t)P * 2, cudaMemcpyHostToDevice);
  for (int r = 0; r < kRanks; ++r) {
    CHECK(cudaMalloc(&d_g[r], (size_t)P * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d_master[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d_m[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d_v[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
  }
  CHECK(zero_init_shards(plan, d_p16, ZERO_BF16, d_master, d_m, d_v, 0xF, NULL) == ZERO_OK,
        "init: %s", zero_last_error());
  /* oracle state */
  float *o_master[kRanks], *o_m[kRanks], *o_v[kRanks];
  for (int r = 0; r < kRanks; ++r) {
    o_master[r] = malloc((size_t)S * 4);
    o_m[r] = calloc((size_t)S, 4);
    o_v[r] = calloc((size_t)S, 4);
    for (int64_t i = 0; i < S; ++i) o_master[r][i] = orc_bf16_to_f32(p16[r * S + i]);
  }
  uint16_t* o_full = calloc((size_t)P, 2);
  zero_adamw_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  orc_hparams ohp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  for (int t = 0; t < 2; ++t) {
    for (int q = 0; q < kRanks; ++q)
      cudaMemcpy(d_g[q], g16[t][q], (size_t)P * 2, cudaMemcpyHostToDevice);
    CHECK(zero_step(plan, (const void* const*)d_g, ZERO_BF16, ZERO_REDUCE_AVG, d_master, d_m, d_v,
                    d_full, NULL, &hp, t + 1, 0xF, 0, NULL) == ZERO_OK,
          "step: %s", zero_last_error());
    CHECK(orc_step(kNumel, kTensors, kRanks, 0, kAlign, 1, 1, (const uint16_t* const*)g16[t],
                   o_master, o_m, o_v, o_full, NULL, &ohp, t + 1, 0xF) == 0, "oracle step");
  }
  CHECK(zero_sync(NULL) == ZERO_OK, "sync: %s", zero_last_error());
  uint16_t* full = malloc((size_t)P * 2);
  cudaMemcpy(full, d_full, (size_t)P * 2, cudaMemcpyDeviceToHost);
  for (int64_t i = 0; i < P; ++i)
    CHECK(full[i] == o_full[i], "full16[%lld]: %04x vs oracle %04x", (long long)i, full[i],
          o_full[i]);
  float* got = malloc((size_t)S * 4);
  for (int r = 0; r < kRanks; ++r) {
    cudaMemcpy(got, d_master[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    for (int64_t i = 0; i < S; ++i) {
      const double a = got[i], b = o_master[r][i];
      const double rel = fabs(a - b) / fmax(fabs(b), 1.1754943508222875e-38);
      CHECK(rel <= 1e-6, "master[%d][%lld]: %.9g vs oracle %.9g", r, (long long)i, a, b);
    }
  }
  printf("gpu ok: %lld elements, 4 virtual ranks, 2 steps match the oracle\n", (long long)P);
  zero_plan_destroy(plan);
  return 0;
}

/* One copy of the optimizer state on the device. */
typedef struct {
  float *master[kRanks], *m[kRanks], *v[kRanks], *gsh[kRanks];
  void *full, *state, *ws;
} DevState;

static int dev_state(DevState* d, zero_plan* plan, void* d_p16, int64_t S, int64_t P,
                     int64_t ws_bytes, const zero_amp_config* cfg) {
  for (int r = 0; r < kRanks; ++r) {
    CHECK(cudaMalloc((void**)&d->master[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d->m[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d->v[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void**)&d->gsh[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
  }
  CHECK(cudaMalloc(&d->full, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&d->state, sizeof(zero_amp_state)) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&d->ws, (size_t)ws_bytes) == cudaSuccess, "cudaMalloc");
  CHECK(zero_init_shards(plan, d_p16, ZERO_BF16, d->master, d->m, d->v, 0xF, NULL) == ZERO_OK,
        "init: %s", zero_last_error());
  CHECK(zero_amp_init(d->state, cfg, NULL) == ZERO_OK, "amp init: %s", zero_last_error());
  return 0;
}

static int amp_checks(void) {
  zero_plan* plan = NULL;
  CHECK(zero_plan_partitions(kNumel, kTensors, kRanks, ZERO_PART_FLAT, kAlign, &plan) == ZERO_OK,
        "plan");
  int64_t phi, P, S, off;
  zero_plan_total(plan, &phi, &P);
  zero_plan_shard(plan, 0, &off, &S);
  const int64_t bucket = 3000;
  const int64_t n_buckets = (P + bucket - 1) / bucket;
  int64_t ws_bytes = 0;
  CHECK(zero_amp_workspace_bytes(plan, 0xF, bucket, &ws_bytes) == ZERO_OK, "workspace bytes");
  uint16_t* p16 = calloc((size_t)P, 2);
  uint16_t* g16[kRanks];
  uint32_t seed = 777u;
  for (int64_t i = 0; i < phi; ++i)
    p16[i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.05f);
  void *d_p16, *d_g[kRanks];
  CHECK(cudaMalloc(&d_p16, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(d_p16, p16, (size_t)P * 2, cudaMemcpyHostToDevice);
  for (int q = 0; q < kRanks; ++q) {
    g16[q] = calloc((size_t)P, 2);
    CHECK(cudaMalloc(&d_g[q], (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  }
  /* loss scale 1, clipping at 0.01 (active), window 2 */
  const zero_amp_config cfg = {1.0, 1.0, 2, 1, 0.01};
  const orc_amp_config ocfg = {1.0, 1.0, 2, 1, 0.01};
  DevState A, B;
  if (dev_state(&A, plan, d_p16, S, P, ws_bytes, &cfg) || dev_state(&B, plan, d_p16, S, P,
                                                                     ws_bytes, &cfg))
    return 1;
  float *o_master[kRanks], *o_m[kRanks], *o_v[kRanks];
  for (int r = 0; r < kRanks; ++r) {
    o_master[r] = malloc((size_t)S * 4);
    o_m[r] = calloc((size_t)S, 4);
    o_v[r] = calloc((size_t)S, 4);
    for (int64_t i = 0; i < S; ++i) o_master[r][i] = orc_bf16_to_f32(p16[r * S + i]);
  }
  uint16_t* o_full = calloc((size_t)P, 2);
  orc_amp_state ost;
  orc_amp_init(&ocfg, &ost);
  const zero_adamw_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  const orc_hparams ohp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  for (int t = 0; t < 3; ++t) {
    for (int q = 0; q < kRanks; ++q) {
      for (int64_t i = 0; i < phi; ++i)
        g16[q][i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.02f);
      cudaMemcpy(d_g[q], g16[q], (size_t)P * 2, cudaMemcpyHostToDevice);
    }
    CHECK(zero_step_amp(plan, (const void* const*)d_g, ZERO_BF16, ZERO_REDUCE_AVG, A.gsh,
                        A.master, A.m, A.v, A.full, NULL, &hp, &cfg, A.state, A.ws, ws_bytes,
                        0xF, bucket, NULL) == ZERO_OK, "step_amp: %s", zero_last_error());
    for (int64_t b = n_buckets - 1; b >= 0; --b)
      CHECK(zero_reduce_scatter_bucket_amp(plan, (const void* const*)d_g, ZERO_BF16,
                                           ZERO_REDUCE_AVG, B.gsh, &hp, B.state, B.ws, ws_bytes,
                                           0xF, bucket, b, NULL) == ZERO_OK,
            "bucket %lld: %s", (long long)b, zero_last_error());
    CHECK(zero_step_amp_reduced(plan, ZERO_BF16, B.gsh, B.master, B.m, B.v, B.full, NULL, &hp,
                                &cfg, B.state, B.ws, ws_bytes, 0xF, bucket, NULL) == ZERO_OK,
          "step_amp_reduced: %s", zero_last_error());
    CHECK(orc_step_amp(kNumel, kTensors, kRanks, 0, kAlign, 1, 1, (const uint16_t* const*)g16,
                       o_master, o_m, o_v, o_full, NULL, &ohp, &ocfg, &ost, 0xF) == 0,
          "oracle step_amp");
  }
  CHECK(zero_sync(NULL) == ZERO_OK, "sync: %s", zero_last_error());
  zero_amp_state sa, sb;
  cudaMemcpy(&sa, A.state, sizeof sa, cudaMemcpyDeviceToHost);
  cudaMemcpy(&sb, B.state, sizeof sb, cudaMemcpyDeviceToHost);
  CHECK(memcmp(&sa, &sb, sizeof sa) == 0, "the two paths' states differ");
  CHECK(sa.step == ost.step && sa.skipped == ost.skipped && sa.scale == ost.scale,
        "state: step %lld scale %g vs oracle %lld %g", (long long)sa.step, sa.scale,
        (long long)ost.step, ost.scale);
  CHECK(fabs(sa.norm - ost.norm) <= 1e-10 * fabs(ost.norm), "norm %.17g vs oracle %.17g",
        sa.norm, ost.norm);
  CHECK(sa.coef < 1.0f, "clipping was not active (coef %g)", (double)sa.coef);
  uint16_t* fa = malloc((size_t)P * 2);
  uint16_t* fb = malloc((size_t)P * 2);
  cudaMemcpy(fa, A.full, (size_t)P * 2, cudaMemcpyDeviceToHost);
  cudaMemcpy(fb, B.full, (size_t)P * 2, cudaMemcpyDeviceToHost);
  CHECK(memcmp(fa, fb, (size_t)P * 2) == 0, "the two paths' parameters differ");
  for (int64_t i = 0; i < P; ++i) {
    const int ka = (fa[i] & 0x8000) ? -(fa[i] & 0x7FFF) : fa[i];
    const int ko = (o_full[i] & 0x8000) ? -(o_full[i] & 0x7FFF) : o_full[i];
    CHECK(abs(ka - ko) <= 1, "full16[%lld]: %04x vs oracle %04x", (long long)i, fa[i],
          o_full[i]);
  }
  float* ga = malloc((size_t)S * 4);
  float* gb = malloc((size_t)S * 4);
  for (int r = 0; r < kRanks; ++r) {
    cudaMemcpy(ga, A.master[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(gb, B.master[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(ga, gb, (size_t)S * 4) == 0, "master[%d] differs between the paths", r);
    for (int64_t i = 0; i < S; ++i) {
      const double a = ga[i], b = o_master[r][i];
      const double rel = fabs(a - b) / fmax(fabs(b), 1.1754943508222875e-38);
      CHECK(rel <= 1e-6, "master[%d][%lld]: %.9g vs oracle %.9g", r, (long long)i, a, b);
    }
  }
  printf("amp ok: %lld elements, %lld buckets reduced last first, 3 clipped steps, both paths "
         "match each other and the oracle\n", (long long)P, (long long)n_buckets);
  zero_plan_destroy(plan);
  return 0;
}

static int offload_checks(void) {
  zero_plan* plan = NULL;
  CHECK(zero_plan_partitions(kNumel, kTensors, kRanks, ZERO_PART_FLAT, kAlign, &plan) == ZERO_OK,
        "plan");
  int64_t phi, P, S, off;
  zero_plan_total(plan, &phi, &P);
  zero_plan_shard(plan, 0, &off, &S);
  uint16_t* p16 = calloc((size_t)P, 2);
  uint16_t* g16[2][kRanks];
  uint32_t seed = 777u;
  for (int64_t i = 0; i < phi; ++i)
    p16[i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.05f);
  for (int t = 0; t < 2; ++t)
    for (int q = 0; q < kRanks; ++q) {
      g16[t][q] = calloc((size_t)P, 2);
      for (int64_t i = 0; i < phi; ++i)
        g16[t][q][i] = orc_f32_to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 0.02f);
    }
  /* device: the replicas and the gathered buffer; host: everything else */
  void *d_full, *d_g[kRanks];
  float *h_master[kRanks], *h_m[kRanks], *h_v[kRanks], *h_gsh[kRanks];
  void* h_s16[kRanks];
  CHECK(cudaMalloc(&d_full, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  for (int r = 0; r < kRanks; ++r) {
    CHECK(cudaMalloc(&d_g[r], (size_t)P * 2) == cudaSuccess, "cudaMalloc");
    CHECK((h_master[r] = aligned_alloc(64, (size_t)S * 4)) != NULL, "aligned_alloc");
    CHECK((h_m[r] = calloc((size_t)S, 4)) != NULL, "calloc");
    CHECK((h_v[r] = calloc((size_t)S, 4)) != NULL, "calloc");
    CHECK(cudaHostAlloc((void**)&h_gsh[r], (size_t)S * 4, cudaHostAllocDefault) == cudaSuccess,
          "cudaHostAlloc");
    CHECK(cudaHostAlloc(&h_s16[r], (size_t)S * 2, cudaHostAllocDefault) == cudaSuccess,
          "cudaHostAlloc");
    for (int64_t i = 0; i < S; ++i) h_master[r][i] = orc_bf16_to_f32(p16[r * S + i]);
  }
  float *o_master[kRanks], *o_m[kRanks], *o_v[kRanks];
  for (int r = 0; r < kRanks; ++r) {
    o_master[r] = malloc((size_t)S * 4);
    o_m[r] = calloc((size_t)S, 4);
    o_v[r] = calloc((size_t)S, 4);
    memcpy(o_master[r], h_master[r], (size_t)S * 4);
  }
  uint16_t* o_full = calloc((size_t)P, 2);
  zero_adamw_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  orc_hparams ohp = {1e-3, 0.9, 0.999, 1e-8, 0.01};
  /* pageable gradient shards are refused before anything is launched */
  float* pageable[kRanks];
  for (int r = 0; r < kRanks; ++r) pageable[r] = h_m[r];
  const int64_t before = zero_launch_count();
  CHECK(zero_offload_step(plan, (const void* const*)d_g, ZERO_BF16, ZERO_REDUCE_AVG, pageable,
                          h_master, h_m, h_v, h_s16, d_full, &hp, 1, 0xF, 1000, 3,
                          NULL) == ZERO_ERR_INVALID, "pageable gradient shards were accepted");
  CHECK(zero_launch_count() == before, "a refused call launched");
  for (int t = 0; t < 2; ++t) {
    for (int q = 0; q < kRanks; ++q)
      cudaMemcpy(d_g[q], g16[t][q], (size_t)P * 2, cudaMemcpyHostToDevice);
    CHECK(zero_offload_step(plan, (const void* const*)d_g, ZERO_BF16, ZERO_REDUCE_AVG, h_gsh,
                            h_master, h_m, h_v, h_s16, d_full, &hp, t + 1, 0xF, 1000, 3,
                            NULL) == ZERO_OK, "offload step: %s", zero_last_error());
    CHECK(orc_step(kNumel, kTensors, kRanks, 0, kAlign, 1, 1, (const uint16_t* const*)g16[t],
                   o_master, o_m, o_v, o_full, NULL, &ohp, t + 1, 0xF) == 0, "oracle step");
  }
  CHECK(zero_sync(NULL) == ZERO_OK, "sync: %s", zero_last_error());
  uint16_t* full = malloc((size_t)P * 2);
  cudaMemcpy(full, d_full, (size_t)P * 2, cudaMemcpyDeviceToHost);
  for (int64_t i = 0; i < P; ++i)
    CHECK(full[i] == o_full[i], "full16[%lld]: %04x vs oracle %04x", (long long)i, full[i],
          o_full[i]);
  for (int r = 0; r < kRanks; ++r) {
    CHECK(memcmp(h_s16[r], o_full + r * S, (size_t)S * 2) == 0, "host shard16[%d]", r);
    for (int64_t i = 0; i < S; ++i) {
      const double a = h_master[r][i], b = o_master[r][i];
      const double rel = fabs(a - b) / fmax(fabs(b), 1.1754943508222875e-38);
      CHECK(rel <= 1e-6, "master[%d][%lld]: %.9g vs oracle %.9g", r, (long long)i, a, b);
    }
  }
  printf("offload ok: %lld elements, host state, chunks of 1000 on 3 host threads, 2 steps "
         "match the oracle\n", (long long)P);
  zero_plan_destroy(plan);
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) return gpu_checks();
  if (argc > 1 && strcmp(argv[1], "amp") == 0) return amp_checks();
  if (argc > 1 && strcmp(argv[1], "offload") == 0) return offload_checks();
  return host_checks();
}
