/*
 * A plain-C caller of the library's ABI (include/zero.h): no Python, no
 * torch.  Mode "host" checks the plan, the memory model and argument
 * rejection (no GPU needed); mode "gpu" allocates device buffers with the
 * CUDA runtime, runs zero_init_shards + two zero_step calls on a small
 * group and compares the results with the CPU oracle, which this test links
 * as a separate library (the two share no code).
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

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) return gpu_checks();
  return host_checks();
}
