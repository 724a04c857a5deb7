// binary16 instantiation of the step kernels.
#include "zero_kernels.cuh"
#include "zero_kernels_tma.cuh"

namespace zero {
template <>
int launch_step_tma<__half>(const LaunchArgs& a, cudaStream_t s) {
  return launch_step_tma_impl<__half>(a, s);
}
template int launch_typed<__half>(Kind, const LaunchArgs&, cudaStream_t);
}  // namespace zero
