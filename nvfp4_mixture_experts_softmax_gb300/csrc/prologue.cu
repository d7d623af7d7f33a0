// Everything before GEMM1 for a small batch, in one block of 1024 threads: reset the device
// status word, max |x| and the activation tensor scale, the NVFP4 encode of x, the router and
// the plan.  For decode-sized batches each of these steps is a few microseconds of launch and
// drain when it runs as its own kernel; here they cost one launch.  The arithmetic is the same
// as in the separate kernels (the quantiser's IEEE divisions, the warp top-k, the stable plan).
#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace nvfp4moe {

namespace {

template <int VPL>
__global__ void __launch_bounds__(kSmallPlanThreads) prologue_small_kernel(const PrologueArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ uint32_t red[32];
  __shared__ float s_ts;
  griddep_wait();
  griddep_launch();
  if (threadIdx.x == 0) *a.status = 0;
  const uint4* x = reinterpret_cast<const uint4*>(a.x);
  const int64_t nvec = (int64_t)a.T * a.H / 8;
  uint32_t m = 0;
  for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) m = max(m, abs_bf16_max8(__ldg(x + i)));
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) {
    if (m >= 0x7F80u) set_status(a.status, MOE_ERR_NONFINITE);
    const float ts = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
    s_ts = ts;
    *a.ts = ts;
  }
  __syncthreads();
  const float ts = s_ts;
  const int64_t nblk = (int64_t)a.T * a.H / 16;
  for (int64_t b = threadIdx.x; b < nblk; b += blockDim.x)
    encode_bf16_block16(x, b, ts, reinterpret_cast<uint2*>(a.xq), a.xsf);
  small_plan_body<VPL>(a.logits, a.T, a.E, a.k, a.shared_rows, a.ids, a.w, a.counts, a.offsets,
                       a.tile_start, a.perm_src, a.perm_w, a.inv, s_dyn);
}

}  // namespace

bool prologue_small_fits(int T, int H, int k) {
  return (int64_t)T * k <= kSmallPlanRows && (int64_t)T * H <= kSmallPrologueElems;
}

cudaError_t launch_prologue_small(const PrologueArgs& a, cudaStream_t s) {
  const size_t smem = small_plan_smem_bytes(a.E);
  const int vpl = (a.E + 31) / 32;
#define NVFP4MOE_PRO(V)                                                                        \
  do {                                                                                         \
    if (smem > 48 * 1024) {                                                                    \
      cudaError_t e = cudaFuncSetAttribute(prologue_small_kernel<V>,                           \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                           (int)smem);                                         \
      if (e != cudaSuccess) return e;                                                          \
    }                                                                                          \
    cudaError_t le = launch_pdl(prologue_small_kernel<V>, dim3(1), dim3(kSmallPlanThreads),    \
                                smem, s, a);                                                   \
    if (le != cudaSuccess) return le;                                                          \
  } while (0)
  if (vpl <= 1) NVFP4MOE_PRO(1);
  else if (vpl <= 2) NVFP4MOE_PRO(2);
  else if (vpl <= 4) NVFP4MOE_PRO(4);
  else if (vpl <= 8) NVFP4MOE_PRO(8);
  else if (vpl <= 16) NVFP4MOE_PRO(16);
  else NVFP4MOE_PRO(kMaxVpl);
#undef NVFP4MOE_PRO
  return cudaGetLastError();
}

}  // namespace nvfp4moe
