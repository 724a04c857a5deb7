// Host-side AdamW of the offloaded optimizer (ZeRO-Offload's CPU optimizer):
// the element loop the host threads of zero_cpu_adamw_shard_step and
// zero_offload_step run.  It performs the same binary32 operations in the
// same order as the GPU update (compiled with -ffp-contract=off, so no
// operation is fused into an FMA; division and square root are the IEEE
// ones), so both give identical bits.  The 16-bit cast is made in the same
// pass, while the updated value is still in a register: the loop streams
// 16 bytes in and 12 + 2 out per element, once.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "zero_host.h"
#include "zero_internal.h"

namespace zero {
namespace {

// Round to nearest even on the upper half of the binary32 pattern; NaN stays
// a quiet NaN with its sign.  Written without a branch so that the loop
// below stays vectorisable.
inline uint16_t to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  const uint32_t rounded = (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
  const uint32_t quiet = (u >> 16) | 0x0040u;
  return static_cast<uint16_t>((u & 0x7fffffffu) > 0x7f800000u ? quiet : rounded);
}

inline uint16_t to_fp16(float x) {
  const _Float16 h = static_cast<_Float16>(x);  // IEEE conversion, nearest even
  uint16_t r;
  memcpy(&r, &h, 2);
  return r;
}

enum Cast { kNoCast, kCastBf16, kCastFp16 };

// kScaled: the gradient is multiplied by `coef` first (one rounding), as the
// mixed-precision update does.
template <Cast C, bool kScaled>
void adamw_loop(const StepScalars& s, float coef, float* __restrict p, float* __restrict m,
                float* __restrict v, const float* __restrict g, uint16_t* __restrict out16,
                int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    const float gi = kScaled ? g[i] * coef : g[i];
    float pp = p[i] * s.d;
    const float mm = s.b1 * m[i] + s.c1 * gi;
    const float vv = s.b2 * v[i] + s.c2 * (gi * gi);
    const float den = sqrtf(vv) / s.sb + s.eps;
    pp = pp - s.ss * (mm / den);
    p[i] = pp;
    m[i] = mm;
    v[i] = vv;
    if (C == kCastBf16) out16[i] = to_bf16(pp);
    if (C == kCastFp16) out16[i] = to_fp16(pp);
  }
}

}  // namespace

namespace {

template <bool kScaled>
void adamw_dispatch(const StepScalars& s, float coef, zero_dtype dtype, float* p, float* m,
                    float* v, const float* g, uint16_t* out16, int64_t n) {
  if (!out16)
    adamw_loop<kNoCast, kScaled>(s, coef, p, m, v, g, nullptr, n);
  else if (dtype == ZERO_BF16)
    adamw_loop<kCastBf16, kScaled>(s, coef, p, m, v, g, out16, n);
  else
    adamw_loop<kCastFp16, kScaled>(s, coef, p, m, v, g, out16, n);
}

}  // namespace

void cpu_adamw_range(const StepScalars& s, zero_dtype dtype, float* p, float* m, float* v,
                     const float* g, uint16_t* out16, int64_t n) {
  adamw_dispatch<false>(s, 1.0f, dtype, p, m, v, g, out16, n);
}

void cpu_adamw_range_scaled(const StepScalars& s, float coef, zero_dtype dtype, float* p,
                            float* m, float* v, const float* g, uint16_t* out16, int64_t n) {
  adamw_dispatch<true>(s, coef, dtype, p, m, v, g, out16, n);
}

}  // namespace zero
