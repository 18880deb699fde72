// bf16 instantiations of the fused gated group-RMSNorm kernels (MAMBA2 only:
// the ONNX contract admits float32 and float16).
#include "ggrn_stream.cuh"

namespace ggrn {
cudaError_t launch_bf16(const KParams& k, const Plan& p, int mode, cudaStream_t s) {
  if (mode == kMamba2) return launch_mode<__nv_bfloat16, kMamba2>(k, p, s);
  return cudaErrorInvalidValue;
}
}  // namespace ggrn

#ifdef GGRN_TIMELINE
// Profiling build only: the timeline stamps of this element type's streaming
// launches (see ggrn_stream.cuh), copied to `host` (64 x 320 x 5 uint64), and
// cleared.
extern "C" int ggrn_timeline_read_bf16(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_ggrn_timeline, sizeof(g_ggrn_timeline)) == cudaSuccess ? 0
                                                                                             : 1;
}
extern "C" int ggrn_timeline_clear_bf16(void) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_ggrn_timeline) != cudaSuccess) return 1;
  return cudaMemset(ptr, 0, sizeof(g_ggrn_timeline)) == cudaSuccess ? 0 : 1;
}
#endif
