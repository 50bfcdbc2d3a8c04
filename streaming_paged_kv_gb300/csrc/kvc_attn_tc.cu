// Tensor-core (tcgen05) paged attention -- not yet enabled.
#include "kvc_internal.h"

namespace kvc {
struct TcMaps {};
bool tc_supported(int, int, int, int) { return false; }
TcMaps* tc_create_maps(void*, int, int, int, int, int, int, cudaError_t* err) {
  if (err) *err = cudaErrorNotSupported;
  return nullptr;
}
void tc_destroy_maps(TcMaps*) {}
cudaError_t launch_attn_tc(const AttnArgs&, TcMaps*, int, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace kvc
