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
  if (a.in_ts) {
    // already quantised input: only its tensor scale is taken over (the permute reads its codes)
    if (threadIdx.x == 0) {
      const float ts = __ldg(a.in_ts);
      if (!(ts >= 0.0f && ts <= 3.402823466e38f)) set_status(a.status, MOE_ERR_NONFINITE);
      *a.ts = ts;
    }
  } else {
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
  }
  small_plan_body<VPL, SQRTSP>(a.logits, a.T, a.E, a.k, a.shared_rows, a.ids, a.w, a.counts,
                               a.offsets, a.tile_start, a.perm_src, a.perm_w, a.inv, s_dyn,
                               a.perm_seg, a.bias);
}

// Decode batches (T <= kDecodeMaxRows = 64): a cluster of kDecodeProCtas CTAs around one cluster
// barrier.
//   A: every thread loads one 16-element block of x, which it keeps in registers for the encode,
//      and takes its max |x|; token t is routed by warp t / C of CTA t % C (C = kDecodeProCtas), the
//      results going to global memory and to the routing CTA's shared memory.
//   B: every CTA combines the partial maxima through distributed shared memory into the tensor
//      scale and gathers the other CTAs' routing results.  Each expert gets the mask of the tokens
//      that chose it (one bit per token: T <= 64), so its count is popcount(mask) and the stable
//      position of token t's assignment to it is offset + popcount(mask & (2^t - 1)): the order of
//      the general plan (expert-major, then assignment order), because a token picks an expert at
//      most once.  Every CTA computes the same plan; CTA 0 alone writes it to global memory.  A table
//      gives each (token, slot) its expert-ordered row and the offset of its scale bytes in the
//      arrangement of the decode GEMM's token operand (tiles of kDecodeTileRows rows: tile = the
//      expert's first tile + rank / kDecodeTileRows, row = rank mod kDecodeTileRows, rank = the
//      row's rank within the expert); then every thread encodes its block once and writes it in
//      token order and to each of the token's expert rows.
// As soon as the segment offsets and tile starts are in global memory, CTA 0 sets a flag that the
// decode GEMM (launched early through programmatic dependent launch) polls before it reads its
// plan, so the weight stream starts while this kernel still encodes; the flag is cleared before
// this grid lets the GEMM launch.
// A CTA keeps its shared memory until the cluster's other CTAs have finished reading it (split
// cluster barrier: arrive after the last remote read, wait before exit).
struct DecodeSmem {
  // byte offsets into the dynamic shared memory
  size_t mask, sfo, ids, w, off, toff, dst, total;
  __host__ __device__ DecodeSmem(int E, int k) {
    const size_t kd = (size_t)k + 1;
    mask = 0;                                                      // u64 [E]
    sfo = mask + 8 * (size_t)E;                                    // i64 [64 * kd]
    ids = sfo + 8 * kDecodeMaxRows * kd;                           // i32 [64 * k]
    w = ids + 4 * (size_t)kDecodeMaxRows * k;                      // f32 [64 * k]
    off = w + 4 * (size_t)kDecodeMaxRows * k;                      // i32 [E + 1]
    toff = off + 4 * ((size_t)E + 1);                              // i32 [E + 1]
    dst = toff + 4 * ((size_t)E + 1);                              // i32 [64 * kd]
    total = dst + 4 * kDecodeMaxRows * kd;
  }
};

template <int VPL, bool SQRTSP>
__global__ void __launch_bounds__(kSmallPlanThreads) decode_prologue_kernel(const DecodePrologueArgs a) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ uint32_t red[32];
  __shared__ uint32_t s_part;
  __shared__ float s_ts;
  griddep_wait();
  // the decode GEMM may start once every CTA of this grid has passed griddep_launch; it reads the
  // plan after polling the flag, which must therefore read 0 until this call's plan is written
  // (the CTA that routes the fewest tokens clears it, off the plan's path)
  if (cluster_ctarank() == kDecodeProCtas - 1) {
    if (threadIdx.x == 0) {
      *a.plan_flag = 0;
      __threadfence();
    }
    __syncthreads();
  }
  griddep_launch();
  constexpr int C = kDecodeProCtas;
  constexpr int nw = kSmallPlanThreads / 32;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* x = reinterpret_cast<const uint4*>(a.x);
  const int T = a.T, E = a.E, k = a.k;
  const int kd = k + 1;   // destinations of a token: its k expert rows, then the shared expert's
  const int R = T * k;
  const int Rt = R + a.shared_rows;
  const int nkb = a.H / 16;
  const DecodeSmem L(E, k);
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(s_dyn + L.mask);
  long long* s_sfo = reinterpret_cast<long long*>(s_dyn + L.sfo);
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_dyn + L.ids);
  float* s_w = reinterpret_cast<float*>(s_dyn + L.w);
  int32_t* s_off = reinterpret_cast<int32_t*>(s_dyn + L.off);
  int32_t* s_toff = reinterpret_cast<int32_t*>(s_dyn + L.toff);
  int32_t* s_dst = reinterpret_cast<int32_t*>(s_dyn + L.dst);
  if (rank == 0 && threadIdx.x == 0) *a.status = 0;
  if (rank == 1 % C)
    for (int i = threadIdx.x; i < a.nready; i += blockDim.x) a.ready[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0ull;

  // ---- A: this thread's first block of x (its load overlaps the routing), routing, max |x| ----
  // (already quantised input: the block's 8 code bytes and its scale byte instead)
  const bool qin = a.in_xq != nullptr;
  const int64_t nblk = (int64_t)T * nkb;
  // 32-block chunks (one per warp: coalesced stores) dealt round robin over the cluster's CTAs,
  // so that a small batch spreads its encode stores over every CTA's memory pipeline instead of
  // loading the first CTA with all of them (T=8: one SM's 20k scattered stores took ~4 us)
  const int64_t bstride = (int64_t)C * blockDim.x;
  const int64_t u0 = ((int64_t)warp * C + rank) * 32 + lane;
  uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
  if (u0 < nblk) {
    if (qin) {
      const uint2 c = __ldg(reinterpret_cast<const uint2*>(a.in_xq) + u0);
      xa = make_uint4(c.x, c.y, (uint32_t)__ldg(a.in_xsf + u0), 0u);
    } else {
      xa = __ldg(x + 2 * u0);
      xb = __ldg(x + 2 * u0 + 1);
    }
  }
  for (int t = warp * C + (int)rank; t < T; t += nw * C) {
    int my_id;
    float my_l;
    warp_topk<VPL, SQRTSP>(a.logits + (int64_t)t * E, E, k, lane, my_id, my_l, a.bias);
    const float w = topk_weight<SQRTSP>(my_l, k, lane);
    if (lane < k) {
      a.ids[(int64_t)t * k + lane] = my_id;
      a.w[(int64_t)t * k + lane] = w;
      s_ids[t * k + lane] = my_id;
      s_w[t * k + lane] = w;
    }
  }
  if (!qin) {
    uint32_t m = max(abs_bf16_max8(xa), abs_bf16_max8(xb));
    for (int64_t u = u0 + bstride; u < nblk; u += bstride)
      m = max(m, max(abs_bf16_max8(__ldg(x + 2 * u)), abs_bf16_max8(__ldg(x + 2 * u + 1))));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) s_part = m;
  }
  cluster_sync();

  // ---- B: tensor scale, every CTA's routing results, token masks per expert ----
  if (qin) {
    if (threadIdx.x == 0) {
      const float ts = __ldg(a.in_ts);
      s_ts = ts;
      if (rank == 0) {
        if (!(ts >= 0.0f && ts <= 3.402823466e38f)) set_status(a.status, MOE_ERR_NONFINITE);
        *a.ts = ts;
      }
    }
  } else if (threadIdx.x < 32) {
    uint32_t m = threadIdx.x < C ? ld_dsmem_u32(&s_part, threadIdx.x) : 0u;
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
    const int t = i / k;
    const uint32_t owner = (uint32_t)(t % C);
    int32_t e = s_ids[i];
    if (owner != rank) {
      e = (int32_t)ld_dsmem_u32(&s_ids[i], owner);
      s_ids[i] = e;
      s_w[i] = __uint_as_float(ld_dsmem_u32(&s_w[i], owner));
    }
    if (e >= 0 && e < E) atomicOr(&s_mask[e], 1ull << t);
  }
  cluster_arrive();   // no remote reads of this cluster after this point
  __syncthreads();

  // counts, offsets and tile starts: one warp, E / 32 consecutive experts per lane
  const bool out = rank == 0;
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(lane * per, E), e1 = min(e0 + per, E);
    int c = 0, tc = 0;
    for (int e = e0; e < e1; ++e) {
      const int n = __popcll(s_mask[e]);
      c += n;
      tc += (n + kDecodeTileRows - 1) / kDecodeTileRows;
    }
    int ci = c, ti = tc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ci, o);
      const int z = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) {
        ci += y;
        ti += z;
      }
    }
    int off = ci - c, toff = ti - tc;
    for (int e = e0; e < e1; ++e) {
      const int n = __popcll(s_mask[e]);
      s_off[e] = off;
      s_toff[e] = toff;
      if (out) {
        if (a.counts) a.counts[e] = n;
        a.offsets[e] = off;
        a.tile_start[e] = toff;
      }
      off += n;
      toff += (n + kDecodeTileRows - 1) / kDecodeTileRows;
    }
    if (lane == 31) {
      s_off[E] = ci;
      s_toff[E] = ti;
      if (out) {
        a.offsets[E] = ci;
        a.tile_start[E] = ti;
        if (a.shared_rows > 0) {
          a.offsets[E + 1] = ci + a.shared_rows;
          a.tile_start[E + 1] = ti + (a.shared_rows + kDecodeTileRows - 1) / kDecodeTileRows;
        }
      }
    }
  }
  __syncthreads();
  // segment offsets and tile starts are in global memory: the decode GEMM may read its plan
  // (a test hook leaves the flag down, so that the GEMM's bounded wait for it runs out)
  if (out && threadIdx.x == 0 && !a.no_plan_flag) {
    __threadfence();
    st_release_s32(a.plan_flag, 1);
  }

  // destination table: expert-ordered row and scale-byte offset of each (token, slot)
  const int wpr = a.H / 64;   // 4-scale words per row
  // tiles of the token-operand scale arrangement: kDecodeTileRows rows of one expert each
  const int ntiles = a.nready;
  for (int i = threadIdx.x; i < T * kd; i += blockDim.x) {
    const int t = i / kd, j = i - t * kd;
    int p = -1, r = 0, tile = 0, e = E;
    if (j < k) {
      e = s_ids[t * k + j];
      if (e >= 0 && e < E) {
        r = __popcll(s_mask[e] & ((1ull << t) - 1ull));
        p = s_off[e] + r;
        tile = s_toff[e] + r / kDecodeTileRows;
      } else {
        set_status(a.status, MOE_ERR_INVALID_ARG);
      }
    } else if (a.shared_rows > 0) {   // the shared expert's rows follow the routed ones
      p = R + t;
      r = t;
      tile = s_toff[E] + r / kDecodeTileRows;
    }
    if (p >= 0 && (p >= Rt || r >= kDecodeMaxRows || tile < 0 || tile >= ntiles)) {
      set_status(a.status, MOE_ERR_INVALID_ARG);
      p = -1;
    }
    if (out && p >= 0) {
      a.perm_src[p] = t;
      a.perm_w[p] = j < k ? s_w[t * k + j] : 1.0f;
      a.perm_seg[p] = e;
      if (j < k) a.inv[t * k + j] = p;
    }
    s_dst[i] = p;
    s_sfo[i] = ((long long)tile * wpr) * 512 + (r % kDecodeTileRows) * 16;
  }
  __syncthreads();

  // ---- encode each (token, block) once into token order and into the token's expert rows ----
  // (quantised input: its blocks are copied into the expert rows as they are)
  const float ts = s_ts;
  for (int64_t u = u0; u < nblk; u += bstride) {
    uint4 v0 = xa, v1 = xb;
    if (u != u0) {
      if (qin) {
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(a.in_xq) + u);
        v0 = make_uint4(c.x, c.y, (uint32_t)__ldg(a.in_xsf + u), 0u);
      } else {
        v0 = __ldg(x + 2 * u);
        v1 = __ldg(x + 2 * u + 1);
      }
    }
    const int t = (int)(u / nkb), b = (int)(u - (int64_t)t * nkb);
    uint32_t lo, hi, sf;
    if (qin) {
      lo = v0.x;
      hi = v0.y;
      sf = v0.z;
    } else {
      quant_bf16_regs16(v0, v1, ts, lo, hi, sf);
      if (a.xq) {
        reinterpret_cast<uint2*>(a.xq)[u] = make_uint2(lo, hi);
        a.xsf[u] = (uint8_t)sf;
      }
    }
    const long long boff = (long long)(b >> 2) * 512 + (b & 3);
    for (int j = 0; j < kd; ++j) {
      const int p = s_dst[t * kd + j];
      if (p < 0) continue;
      *reinterpret_cast<uint2*>(a.xq_perm + (size_t)p * (a.H / 2) + (size_t)b * 8) =
          make_uint2(lo, hi);
      a.xsf_tiles[s_sfo[t * kd + j] + boff] = (uint8_t)sf;
    }
  }
  cluster_wait();
}

}  // namespace

cudaError_t launch_decode_prologue(const DecodePrologueArgs& a, cudaStream_t s) {
  if (a.T > kDecodeMaxRows || a.k > 32) return cudaErrorInvalidValue;
  const size_t smem = DecodeSmem(a.E, a.k).total;
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
