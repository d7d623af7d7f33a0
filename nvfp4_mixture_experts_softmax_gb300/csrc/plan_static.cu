// moe_plan_static: the router + plan of moe_plan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: a plugin running inside a host
// framework that owns every device allocation, code that runs while a memory pool is frozen or
// capped, or a thin C caller with no allocator of its own.  This entry point therefore keeps its
// scratch in a file-scope static device array of a fixed size.  Every GPU that loads the library
// reserves that array until the process exits.  The array's address is looked up with
// cudaGetSymbolAddress once per device (on that device's first call), because in host code the
// array's name is only a host-side stand-in, not a device address.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticPlanScratchBytes = MOE_PLAN_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_plan_scratch[kStaticPlanScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_plan_scratch on the current device (looked up once per device).
int scratch_on_current_device(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
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
  const int st = scratch_on_current_device(&scratch);
  if (st != MOE_OK) return st;
  // The plan clears the status word at the start of every call and overwrites every histogram
  // and base entry it later reads, so nothing left over from the previous call is used.
  return moe_plan(logits, T, E, k, topk_ids, topk_w, counts, offsets, perm_src, inv, scratch,
                  kStaticPlanScratchBytes, stream);
}
