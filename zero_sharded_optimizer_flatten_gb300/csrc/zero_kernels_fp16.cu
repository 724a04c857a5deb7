// binary16 instantiation of the step kernels.
#include "zero_kernels.cuh"

namespace zero {
template int launch_typed<__half>(Kind, const LaunchArgs&, cudaStream_t);
}  // namespace zero
