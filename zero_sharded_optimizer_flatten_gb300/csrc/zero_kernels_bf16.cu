// bfloat16 instantiation of the step kernels.
#include "zero_kernels.cuh"
#include "zero_kernels_tma.cuh"

namespace zero {
template <>
int launch_step_tma<__nv_bfloat16>(const LaunchArgs& a, cudaStream_t s) {
  return launch_step_tma_impl<__nv_bfloat16>(a, s);
}
template int launch_typed<__nv_bfloat16>(Kind, const LaunchArgs&, cudaStream_t);
}  // namespace zero
