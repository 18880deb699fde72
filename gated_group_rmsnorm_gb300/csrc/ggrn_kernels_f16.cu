// fp16 instantiations of the fused gated group-RMSNorm kernels.
#include "ggrn_stream.cuh"

namespace ggrn {
cudaError_t launch_f16(const KParams& k, const Plan& p, int mode, cudaStream_t s) {
  if (mode == kMamba2) return launch_mode<__half, kMamba2>(k, p, s);
  if (mode == kOnnx) return launch_mode<__half, kOnnx>(k, p, s);
  return cudaErrorInvalidValue;
}
}  // namespace ggrn
