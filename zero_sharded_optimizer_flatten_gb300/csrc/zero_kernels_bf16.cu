// bfloat16 instantiation of the step kernels.
#include "zero_kernels.cuh"

namespace zero {
template int launch_typed<__nv_bfloat16>(Kind, const LaunchArgs&, cudaStream_t);
}  // namespace zero
