// Host-side optimizer loop of the offloaded mixed-precision step (no device
// code; the unscaled loop is declared beside the kernels' shared types).
#pragma once

#include <stdint.h>

#include "zero_internal.h"

namespace zero {

// AdamW + cast over n elements of host memory with the gradient multiplied
// by coef first (one binary32 rounding), as the mixed-precision update
// kernel does (zero_cpu_adam.cpp).  out16 may be NULL (no cast).
void cpu_adamw_range_scaled(const StepScalars& s, float coef, zero_dtype dtype, float* p,
                            float* m, float* v, const float* g, uint16_t* out16, int64_t n);

}  // namespace zero
