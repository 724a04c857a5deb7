// Status and error-message helpers shared by the C-ABI translation units.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <stdarg.h>
#include <stdio.h>

#include "zero.h"

namespace zero {

// Thread-local message of the last failed call (see zero_last_error).
char* error_buffer();

inline void clear_error() { error_buffer()[0] = '\0'; }

#if defined(__GNUC__)
__attribute__((format(printf, 2, 3)))
#endif
inline zero_status fail(zero_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(error_buffer(), 1024, fmt, ap);
  va_end(ap);
  return st;
}

// An NVTX range named after the C-ABI call, for timelines in Nsight tools
// (a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace zero
