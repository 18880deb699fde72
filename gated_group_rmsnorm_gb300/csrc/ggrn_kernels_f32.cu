// f32 instantiations of the fused gated group-RMSNorm kernels.
#include "ggrn_stream.cuh"

namespace ggrn {
cudaError_t launch_f32(const KParams& k, const Plan& p, int mode, cudaStream_t s) {
  if (mode == kMamba2) return launch_mode<float, kMamba2>(k, p, s);
  if (mode == kOnnx) return launch_mode<float, kOnnx>(k, p, s);
  return cudaErrorInvalidValue;
}
}  // namespace ggrn

#ifdef GGRN_TIMELINE
// Profiling build only: the timeline stamps of this element type's streaming
// launches (see ggrn_stream.cuh), copied to `host` (64 x 320 x 5 uint64), and
// cleared.
extern "C" int ggrn_timeline_read_f32(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_ggrn_timeline, sizeof(g_ggrn_timeline)) == cudaSuccess ? 0
                                                                                             : 1;
}
extern "C" int ggrn_timeline_clear_f32(void) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_ggrn_timeline) != cudaSuccess) return 1;
  return cudaMemset(ptr, 0, sizeof(g_ggrn_timeline)) == cudaSuccess ? 0 : 1;
}
#endif
