// moe_plan_static: the router + plan of moe_plan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: a plugin running inside a host
// framework that owns every device allocation, code that runs while a memory pool is frozen or
// capped, or a thin C caller with no allocator of its own.  This entry point therefore keeps its
// scratch in a file-scope static device array of a fixed size.  Every GPU that loads the library
// reserves that array until the process exits.  In host code the array's name is only a
// host-side stand-in, not a device address, so the address is looked up with
// cudaGetSymbolAddress, with the target device current.
//
// The lookup is repeated on every call that is not being recorded into a CUDA graph: a device
// reset (cudaDeviceReset, or a reset of the primary context by another runtime in the process)
// reloads the module and may move the array, and a cached address would then point at freed
// memory.  A call made during stream capture cannot take that lookup safely (it may load the
// module, which capture forbids), so it uses the address found by the last uncaptured call on
// the same device: the first call on a device, and the first call after a reset, must come before
// any capture.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticPlanScratchBytes = MOE_PLAN_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_plan_scratch[kStaticPlanScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};   // address found by the last uncaptured call per device

// Device address of g_plan_scratch on the current device.
int scratch_on_current_device(cudaStream_t s, uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (g_scratch_ptr[dev] == nullptr) {
    return MOE_ERR_CUDA;   // never looked up outside a capture on this device
  }
  *out = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  return MOE_OK;
}

}  // namespace

extern "C" int moe_plan_static(const float* logits, int32_t T, int32_t E, int32_t k,
                               int32_t* topk_ids, float* topk_w, int32_t* counts,
                               int32_t* offsets, int32_t* perm_src, int32_t* inv,
                               moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  const size_t need = moe_plan_workspace_size(T, E, k);
  if (need == 0 || need > kStaticPlanScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* scratch = nullptr;
  const int st = scratch_on_current_device(reinterpret_cast<cudaStream_t>(stream), &scratch);
  if (st != MOE_OK) return st;
  // The plan clears the status word at the start of every call and overwrites every histogram
  // and base entry it later reads, so nothing left over from the previous call is used.
  return moe_plan(logits, T, E, k, topk_ids, topk_w, counts, offsets, perm_src, inv, scratch,
                  kStaticPlanScratchBytes, stream);
}
