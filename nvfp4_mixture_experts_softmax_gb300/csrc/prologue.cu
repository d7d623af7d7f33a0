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

template <int VPL, bool SQRTSP>
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
  small_plan_body<VPL, SQRTSP>(a.logits, a.T, a.E, a.k, a.shared_rows, a.ids, a.w, a.counts,
                               a.offsets, a.tile_start, a.perm_src, a.perm_w, a.inv, s_dyn,
                               a.perm_seg, a.bias);
}

// Decode batches (T <= kDecodeMaxRows): a cluster of kDecodeProCtas CTAs in two phases around
// one cluster barrier.
//   A: one warp per token routes (top-k + weights, written to global memory and to the routing
//      CTA's shared memory) while every CTA reduces max |x| over its slice of x;
//   B: every CTA combines the partial maxima through distributed shared memory into the tensor
//      scale, gathers the other CTAs' routing results the same way and places all assignments
//      itself (the same stable plan in every CTA; CTA 0 alone writes it to global memory).  Then
//      one thread per (token, 16-element block) encodes the block once and writes it in token
//      order and into each of the token's expert-ordered rows: the codes into xq_perm, the
//      scale byte into the 32x4x4 arrangement of the decode GEMM's token operand (tile = the
//      expert's tile index, row = expert-ordered row - the expert's offset).
// A CTA keeps its shared memory until the cluster's other CTAs have finished reading it (split
// cluster barrier: arrive after the last remote read, wait before exit).
template <int VPL, bool SQRTSP>
__global__ void __launch_bounds__(kSmallPlanThreads) decode_prologue_kernel(const DecodePrologueArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ uint32_t red[32];
  __shared__ uint32_t s_part;
  __shared__ float s_ts;
  griddep_wait();
  griddep_launch();
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kSmallPlanThreads / 32;
  const uint4* x = reinterpret_cast<const uint4*>(a.x);
  const int R = a.T * a.k;
  const int Rt = R + a.shared_rows;
  const int nkb = a.H / 16;
  // small_place's scratch, then the per-assignment expert-ordered row and the per-expert tile
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_dyn) + 3 * a.E;
  float* s_w = reinterpret_cast<float*>(s_ids + kSmallPlanRows);
  int32_t* s_off = reinterpret_cast<int32_t*>(s_dyn) + a.E;
  int32_t* s_inv = reinterpret_cast<int32_t*>(s_dyn + small_plan_smem_bytes(a.E));
  int32_t* s_toff = s_inv + kSmallPlanRows;
  if (rank == 0 && threadIdx.x == 0) *a.status = 0;

  // ---- A: routing (warp per token) and partial max |x| ----
  // the first two activation vectors of each thread are loaded before the routing so that their
  // memory latency overlaps the logits'
  const int64_t nvec = (int64_t)a.T * a.H / 8;
  const int64_t vstride = (int64_t)kDecodeProCtas * blockDim.x;
  const int64_t v0 = (int64_t)rank * blockDim.x + threadIdx.x;
  uint4 xv0 = make_uint4(0u, 0u, 0u, 0u), xv1 = make_uint4(0u, 0u, 0u, 0u);
  if (v0 < nvec) xv0 = __ldg(x + v0);
  if (v0 + vstride < nvec) xv1 = __ldg(x + v0 + vstride);
  for (int t = (int)rank * nw + warp; t < a.T; t += kDecodeProCtas * nw) {
    int my_id;
    float my_l;
    warp_topk<VPL, SQRTSP>(a.logits + (int64_t)t * a.E, a.E, a.k, lane, my_id, my_l, a.bias);
    const float w = topk_weight<SQRTSP>(my_l, a.k, lane);
    if (lane < a.k) {
      a.ids[(int64_t)t * a.k + lane] = my_id;
      a.w[(int64_t)t * a.k + lane] = w;
      s_ids[t * a.k + lane] = my_id;
      s_w[t * a.k + lane] = w;
    }
  }
  {
    uint32_t m = max(abs_bf16_max8(xv0), abs_bf16_max8(xv1));
    for (int64_t i = v0 + 2 * vstride; i < nvec; i += vstride) m = max(m, abs_bf16_max8(__ldg(x + i)));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) s_part = m;
  }
  cluster_sync();

  // ---- B: tensor scale and routing results from every CTA, then the plan in every CTA ----
  if (threadIdx.x < 32) {
    uint32_t m = threadIdx.x < kDecodeProCtas ? ld_dsmem_u32(&s_part, threadIdx.x) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) {
      const float ts = __fdiv_rn(bf16_bits_to_f32(m), 2688.0f);
      s_ts = ts;
      if (rank == 0) {
        if (m >= 0x7F80u) set_status(a.status, MOE_ERR_NONFINITE);
        *a.ts = ts;
      }
    }
  }
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    const uint32_t owner = (uint32_t)((i / a.k) / nw) % kDecodeProCtas;   // CTA that routed token
    if (owner != rank) {
      s_ids[i] = (int32_t)ld_dsmem_u32(&s_ids[i], owner);
      s_w[i] = __uint_as_float(ld_dsmem_u32(&s_w[i], owner));
    }
  }
  cluster_arrive();   // no remote reads of this cluster after this point
  int32_t* s_cnt = reinterpret_cast<int32_t*>(s_dyn);
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    const int e = s_ids[i];
    if (e >= 0 && e < a.E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  const bool out = rank == 0;
  small_place(a.T, a.E, a.k, a.shared_rows, out ? a.counts : nullptr, out ? a.offsets : nullptr,
              out ? a.tile_start : nullptr, out ? a.perm_src : nullptr, out ? a.perm_w : nullptr,
              out ? a.inv : nullptr, s_dyn, out ? a.perm_seg : nullptr, s_inv, s_toff);
  __syncthreads();
  const float ts = s_ts;

  // ---- encode each (token, block) once into token order and into the token's expert rows ----
  const int wpr = a.H / 64;   // 4-scale words per row
  const int64_t nblk = (int64_t)a.T * nkb;
  for (int64_t u = (int64_t)rank * blockDim.x + threadIdx.x; u < nblk;
       u += (int64_t)kDecodeProCtas * blockDim.x) {
    const int t = (int)(u / nkb), b = (int)(u - (int64_t)t * nkb);
    uint32_t lo, hi, sf;
    quant_bf16_block16(x, u, ts, lo, hi, sf);
    reinterpret_cast<uint2*>(a.xq)[u] = make_uint2(lo, hi);
    a.xsf[u] = (uint8_t)sf;
    for (int j = 0; j <= a.k; ++j) {
      int p, r, tile;
      if (j < a.k) {
        const int e = s_ids[t * a.k + j];
        if (e < 0 || e >= a.E) {
          set_status(a.status, MOE_ERR_INVALID_ARG);
          continue;
        }
        p = s_inv[t * a.k + j];
        r = p - s_off[e];
        tile = s_toff[e];
      } else {
        if (a.shared_rows == 0) break;
        p = R + t;        // the shared expert's rows follow the routed ones, in token order
        r = t;
        tile = s_toff[a.E];
      }
      if (p < 0 || p >= Rt || r < 0 || r >= kDecodeMaxRows || tile < 0 || tile > Rt) {
        set_status(a.status, MOE_ERR_INVALID_ARG);
        continue;
      }
      *reinterpret_cast<uint2*>(a.xq_perm + (size_t)p * (a.H / 2) + (size_t)b * 8) =
          make_uint2(lo, hi);
      a.xsf_tiles[((size_t)tile * wpr + b / 4) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (b & 3)] =
          (uint8_t)sf;
    }
  }
  cluster_wait();
}

}  // namespace

cudaError_t launch_decode_prologue(const DecodePrologueArgs& a, cudaStream_t s) {
  // small_place's scratch + expert-ordered row per assignment + first tile per segment
  const size_t smem = small_plan_smem_bytes(a.E) + sizeof(int32_t) * (kSmallPlanRows + a.E + 1);
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
#define NVFP4MOE_DPRO2(V, SP)                                                                  \
  do {                                                                                         \
    if (smem > 48 * 1024) {                                                                    \
      cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<V, SP>,                      \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                           (int)smem);                                         \
      if (e != cudaSuccess) return e;                                                          \
    }                                                                                          \
    return cudaLaunchKernelEx(&cfg, decode_prologue_kernel<V, SP>, a);                         \
  } while (0)
#define NVFP4MOE_DPRO(V)                                                                       \
  do {                                                                                         \
    if (a.sqrtsp) NVFP4MOE_DPRO2(V, true);                                                     \
    else NVFP4MOE_DPRO2(V, false);                                                             \
  } while (0)
  if (vpl <= 1) NVFP4MOE_DPRO(1);
  else if (vpl <= 2) NVFP4MOE_DPRO(2);
  else if (vpl <= 4) NVFP4MOE_DPRO(4);
  else if (vpl <= 8) NVFP4MOE_DPRO(8);
  else if (vpl <= 16) NVFP4MOE_DPRO(16);
  else NVFP4MOE_DPRO(kMaxVpl);
#undef NVFP4MOE_DPRO
#undef NVFP4MOE_DPRO2
}

bool prologue_small_fits(int T, int H, int k) {
  return (int64_t)T * k <= kSmallPlanRows && (int64_t)T * H <= kSmallPrologueElems;
}

cudaError_t launch_prologue_small(const PrologueArgs& a, cudaStream_t s) {
  const size_t smem = small_plan_smem_bytes(a.E);
  const int vpl = (a.E + 31) / 32;
#define NVFP4MOE_PRO2(V, SP)                                                                   \
  do {                                                                                         \
    if (smem > 48 * 1024) {                                                                    \
      cudaError_t e = cudaFuncSetAttribute(prologue_small_kernel<V, SP>,                       \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                           (int)smem);                                         \
      if (e != cudaSuccess) return e;                                                          \
    }                                                                                          \
    cudaError_t le = launch_pdl(prologue_small_kernel<V, SP>, dim3(1), dim3(kSmallPlanThreads), \
                                smem, s, a);                                                   \
    if (le != cudaSuccess) return le;                                                          \
  } while (0)
#define NVFP4MOE_PRO(V)                                                                        \
  do {                                                                                         \
    if (a.sqrtsp) NVFP4MOE_PRO2(V, true);                                                      \
    else NVFP4MOE_PRO2(V, false);                                                              \
  } while (0)
  if (vpl <= 1) NVFP4MOE_PRO(1);
  else if (vpl <= 2) NVFP4MOE_PRO(2);
  else if (vpl <= 4) NVFP4MOE_PRO(4);
  else if (vpl <= 8) NVFP4MOE_PRO(8);
  else if (vpl <= 16) NVFP4MOE_PRO(16);
  else NVFP4MOE_PRO(kMaxVpl);
#undef NVFP4MOE_PRO
#undef NVFP4MOE_PRO2
  return cudaGetLastError();
}

}  // namespace nvfp4moe
