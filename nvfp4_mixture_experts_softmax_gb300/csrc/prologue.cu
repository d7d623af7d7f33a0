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
                       a.tile_start, a.perm_src, a.perm_w, a.inv, s_dyn, a.perm_seg);
}

// Decode batches (T <= kDecodeMaxRows): a cluster of kDecodeProCtas CTAs in three phases
// separated by cluster barriers.
//   A: one warp per token routes (top-k + weights, written to global memory) while every CTA
//      reduces max |x| over its slice of x into its shared memory;
//   B: every CTA combines the partial maxima through distributed shared memory into the tensor
//      scale; CTA 0 counts, scans and places the assignments (the plan); the other CTAs encode
//      x in token order, one thread per 16-element block;
//   C: all CTAs copy each permuted row p from token perm_src[p] into xq_perm (16-byte vectors)
//      and its scale words into the 32x4x4 arrangement of the decode GEMM's token operand
//      (tile = the expert's tile index, row = p - offsets[expert]).
template <int VPL>
__global__ void __launch_bounds__(kSmallPlanThreads) decode_prologue_kernel(const DecodePrologueArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ uint32_t red[32];
  __shared__ uint32_t s_part;
  griddep_wait();
  griddep_launch();
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kSmallPlanThreads / 32;
  const uint4* x = reinterpret_cast<const uint4*>(a.x);
  const int R = a.T * a.k;
  const int Rt = R + a.shared_rows;
  const int nkb = a.H / 16;

  // ---- A: routing (warp per token) and partial max |x| ----
  for (int t = (int)rank * nw + warp; t < a.T; t += kDecodeProCtas * nw) {
    int my_id;
    float my_l;
    warp_topk<VPL>(a.logits + (int64_t)t * a.E, a.E, a.k, lane, my_id, my_l);
    const float w = topk_weight(my_l, a.k, lane);
    if (lane < a.k) {
      a.ids[(int64_t)t * a.k + lane] = my_id;
      a.w[(int64_t)t * a.k + lane] = w;
    }
  }
  {
    const int64_t nvec = (int64_t)a.T * a.H / 8;
    uint32_t m = 0;
    for (int64_t i = (int64_t)rank * blockDim.x + threadIdx.x; i < nvec;
         i += (int64_t)kDecodeProCtas * blockDim.x)
      m = max(m, abs_bf16_max8(__ldg(x + i)));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) s_part = m;
  }
  cluster_sync();

  // ---- B: tensor scale; plan (CTA 0) | token-order encode (CTAs 1..) ----
  __shared__ float s_ts;
  if (threadIdx.x < 32) {
    uint32_t m = threadIdx.x < kDecodeProCtas ? ld_dsmem_u32(&s_part, threadIdx.x) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) {
      const float ts = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
      s_ts = ts;
      if (rank == 0) {
        *a.status = 0;
        if (m >= 0x7F80u) set_status(a.status, MOE_ERR_NONFINITE);
        *a.ts = ts;
      }
    }
  }
  __syncthreads();
  const float ts = s_ts;
  if (rank == 0) {
    int32_t* s_cnt = reinterpret_cast<int32_t*>(s_dyn);
    int32_t* s_ids = s_cnt + 3 * a.E;
    float* s_w = reinterpret_cast<float*>(s_ids + kSmallPlanRows);
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
      const int e = __ldcg(a.ids + i);   // written in phase A by other CTAs
      s_ids[i] = e;
      s_w[i] = __ldcg(a.w + i);
      if (e >= 0 && e < a.E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    small_place(a.T, a.E, a.k, a.shared_rows, a.counts, a.offsets, a.tile_start, a.perm_src,
                a.perm_w, a.inv, s_dyn, a.perm_seg);
  } else {
    const int64_t nblk = (int64_t)a.T * nkb;
    for (int64_t b = (int64_t)(rank - 1) * blockDim.x + threadIdx.x; b < nblk;
         b += (int64_t)(kDecodeProCtas - 1) * blockDim.x)
      encode_bf16_block16(x, b, ts, reinterpret_cast<uint2*>(a.xq), a.xsf);
  }
  cluster_sync();

  // ---- C: expert-ordered copy of the codes and the arranged scale words ----
  const int vec_per_row = a.H / 32;     // 16-byte vectors of codes per row
  const int64_t nvec_c = (int64_t)Rt * vec_per_row;
  const int64_t stride = (int64_t)kDecodeProCtas * blockDim.x;
  for (int64_t i = (int64_t)rank * blockDim.x + threadIdx.x; i < nvec_c; i += stride) {
    const int p = (int)(i / vec_per_row), v = (int)(i - (int64_t)p * vec_per_row);
    const int t = __ldcg(a.perm_src + p);
    if (t < 0 || t >= a.T) {
      set_status(a.status, MOE_ERR_INVALID_ARG);
      continue;
    }
    const uint4 c = __ldcg(reinterpret_cast<const uint4*>(a.xq + (size_t)t * (a.H / 2)) + v);
    reinterpret_cast<uint4*>(a.xq_perm + (size_t)p * (a.H / 2))[v] = c;
  }
  const int wpr = a.H / 64;             // 4-scale words per row
  const int64_t nw_c = (int64_t)Rt * wpr;
  for (int64_t i = (int64_t)rank * blockDim.x + threadIdx.x; i < nw_c; i += stride) {
    const int p = (int)(i / wpr), wd = (int)(i - (int64_t)p * wpr);
    const int t = __ldcg(a.perm_src + p);
    const int e = __ldcg(a.perm_seg + p);
    if (t < 0 || t >= a.T || e < 0 || e > a.E) {
      set_status(a.status, MOE_ERR_INVALID_ARG);
      continue;
    }
    const int r = p - __ldcg(a.offsets + e);
    const int tile = __ldcg(a.tile_start + e);
    if (r < 0 || r >= kDecodeMaxRows) {
      set_status(a.status, MOE_ERR_INVALID_ARG);
      continue;
    }
    const uint32_t word = __ldcg(reinterpret_cast<const uint32_t*>(a.xsf + (size_t)t * nkb) + wd);
    *reinterpret_cast<uint32_t*>(a.xsf_tiles + ((size_t)tile * wpr + wd) * 512 + (r & 31) * 16 +
                                 (r >> 5) * 4) = word;
  }
}

}  // namespace

cudaError_t launch_decode_prologue(const DecodePrologueArgs& a, cudaStream_t s) {
  const size_t smem = small_plan_smem_bytes(a.E);
  const int vpl = (a.E + 31) / 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kDecodeProCtas);
  cfg.blockDim = dim3(kSmallPlanThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kDecodeProCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
#define NVFP4MOE_DPRO(V)                                                                       \
  do {                                                                                         \
    if (smem > 48 * 1024) {                                                                    \
      cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<V>,                          \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                           (int)smem);                                         \
      if (e != cudaSuccess) return e;                                                          \
    }                                                                                          \
    return cudaLaunchKernelEx(&cfg, decode_prologue_kernel<V>, a);                             \
  } while (0)
  if (vpl <= 1) NVFP4MOE_DPRO(1);
  else if (vpl <= 2) NVFP4MOE_DPRO(2);
  else if (vpl <= 4) NVFP4MOE_DPRO(4);
  else if (vpl <= 8) NVFP4MOE_DPRO(8);
  else if (vpl <= 16) NVFP4MOE_DPRO(16);
  else NVFP4MOE_DPRO(kMaxVpl);
#undef NVFP4MOE_DPRO
}

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
