// f32 instantiations of the fused gated group-RMSNorm kernels.
#include "ggrn_stream.cuh"

namespace ggrn {
cudaError_t launch_f32(const KParams& k, const Plan& p, int mode, cudaStream_t s) {
  if (mode == kMamba2) return launch_mode<float, kMamba2>(k, p, s);
  if (mode == kOnnx) return launch_mode<float, kOnnx>(k, p, s);
  return cudaErrorInvalidValue;
}
}  // namespace ggrn
