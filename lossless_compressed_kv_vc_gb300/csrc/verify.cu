// Verification attention (placeholder until the tensor-core kernel lands).
#include "vc_internal.cuh"

namespace vc {
size_t verify_workspace_size(const vc_shape* shape, int32_t max_rows) { return 0; }
cudaError_t launch_verify(const vc_shape* shape, const vc_verify_req* req, void* ws, size_t ws_bytes,
                          int32_t* dev_status, cudaStream_t stream, vc_status* st) {
  *st = VC_ERR_UNSUPPORTED;
  return cudaSuccess;
}
}  // namespace vc
