// vc_draft_attn_noalloc: the draft step for callers that cannot allocate device memory.
//
// vc_draft_attn needs a caller-provided workspace for its per-split partial results. Some callers
// cannot provide one: a plugin whose host application owns every device allocation and hands it
// no allocator, or a serving loop that must never call cudaMalloc/cudaFree because those calls can
// synchronise the whole device and stall every other stream. This entry point uses a fixed scratch
// array compiled into the library instead, and allocates nothing.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it until
// the process exits. In host code its name is only a host-side stand-in, so its device address is
// looked up once per device with cudaGetSymbolAddress (on the first call made with that device
// current) and cached; that first call also zero-fills the array on the caller's stream (the
// draft kernel's arrival counters start at zero and every call returns them to zero). All calls
// share the array and it keeps the last call's contents. The counters occupy a block at the start
// whose size and place do not depend on the call's shape, so a call with more KV heads than the
// one before finds zero counters, not the earlier call's partials; the draft kernels write every
// partial before reading it. Calls that overlap on the GPU (different streams, or graph replays
// running concurrently) race on it.
#include "vc_internal.cuh"

#include <mutex>

namespace {

constexpr size_t kScratchBytes = VC_DRAFT_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_draft_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" vc_status vc_draft_attn_noalloc(const vc_shape* shape, const vc_draft_req* req, int32_t* dev_status,
                                           cudaStream_t stream) {
  const size_t need = vc_workspace_size(VC_CALL_DRAFT, shape, 0);
  if (need == 0) return VC_ERR_INVALID;          // malformed shape
  if (need > kScratchBytes) return VC_ERR_WORKSPACE;  // larger than the static scratch
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VC_ERR_CUDA;
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ptr = g_scratch_ptr[dev];
    if (!ptr) {
      if (cudaGetSymbolAddress(&ptr, g_draft_scratch) != cudaSuccess || !ptr ||
          cudaMemsetAsync(ptr, 0, kScratchBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_CUDA;
      }
      g_scratch_ptr[dev] = ptr;
    }
  }
  return vc_draft_attn(shape, req, ptr, kScratchBytes, dev_status, stream);
}
