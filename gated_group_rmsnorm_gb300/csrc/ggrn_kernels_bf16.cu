// bf16 instantiations of the fused gated group-RMSNorm kernels (MAMBA2 only:
// the ONNX contract admits float32 and float16).
#include "ggrn_stream.cuh"

namespace ggrn {
cudaError_t launch_bf16(const KParams& k, const Plan& p, int mode, cudaStream_t s) {
  if (mode == kMamba2) return launch_mode<__nv_bfloat16, kMamba2>(k, p, s);
  return cudaErrorInvalidValue;
}
}  // namespace ggrn
