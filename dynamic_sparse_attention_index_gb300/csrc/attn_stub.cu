// Placeholder attention launchers (replaced by the tcgen05 kernels).
#include "common.cuh"

namespace vs {
size_t attn_fwd_ws_bytes(const vs_params&) { return 256; }
size_t attn_bwd_ws_bytes(const vs_params&) { return 256; }
cudaError_t launch_attn_fwd(const vs_params&, const vs_index&, const void*, const void*, const void*, void*, float*,
                            void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_attn_bwd(const vs_params&, const vs_index&, const void*, const void*, const void*, const void*,
                            const float*, const void*, void*, void*, void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace vs
