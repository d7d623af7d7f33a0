// Grouped block-scaled FP4 GEMM for decode-sized batches (every expert receives at most 64 rows),
// with the operands swapped: the expert's weights are the MMA's A operand (M = 128 weight rows of
// one packed block per K stage, loaded by one bulk copy) and the expert's token rows are the
// B operand (N = the rows rounded up to 16).  The tensor core then works on the real tokens
// only, a pipeline stage is 28 KB instead of 36 KB (7 stages in flight), and the accumulator
// holds one weight row per TMEM lane and one token per column:
//   GEMM1 (mode 0): warp w of the epilogue holds the 16 gate rows and the 16 up rows of one
//          16-feature NVFP4 block, so each half-warp computes silu(g)*u of one token and
//          requantises the block with half-warp reductions;
//   GEMM2 (mode 1 / 2): lanes hold consecutive output features, so a token's row is written (or
//          reduced) 128 contiguous bytes per warp.
// Every operand arrives by the copy engine: per stage one bulk copy of the weight block, one
// 2-D TMA tile (128-byte swizzle) of the expert's token rows - the activations (GEMM1) or h
// (GEMM2) are stored in expert order, so an expert's rows are contiguous - and one bulk copy of
// the tokens' scales, which the producer kernels write pre-arranged per expert tile.  Warps:
// 0-3 epilogue, 4 copy issue, 5 MMA, 6 scale factors ("nvfp4-megamoe-kernel compare
// pre-b1...master", section "MoE kernel": TMA, MMA and epilogue warps; the pages keep decode on
// 1-CTA tiles).  The eight shared -> tensor memory scale copies of a stage hold up the thread that
// issues them for a long time, so a warp of their own issues them one stage ahead of the MMA
// thread and signals it through an mbarrier; the MMA thread then issues only the four MMAs of a
// stage, with descriptors advanced by additions.  Three TMEM accumulators let the epilogue trail
// the main loop by up to two tiles.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kStages = 7;
constexpr int kAccBufs = 3;
constexpr int kXBoxRows = 16;                          // token rows per TMA box
constexpr int kEpiWarps = 4;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSfWarp = 6;
constexpr int kThreads = (kSfWarp + 1) * 32;
constexpr int kNmax = kDecodeMaxRows;                 // token rows per expert tile
constexpr int kXOff = kTileBlockBytes;                 // token codes after the weight block
constexpr int kXBytes = kNmax * 128;
constexpr int kXSfOff = kXOff + kXBytes;               // token scales
constexpr int kXSfBytes = 4 * 512;
constexpr int kStageBytes = kXSfOff + kXSfBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kNmax;
constexpr uint32_t kSfCol0 = kAccBufs * kAccCols;
constexpr uint32_t kSfColsPerStage = 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(kStageBytes % 1024 == 0 && kXOff % 1024 == 0, "1024-byte aligned swizzled tiles");
static_assert(kStages * kStageBytes + 1024 + 256 + 8 * 1027 <= 232448, "shared memory");
static_assert((3 * kStages + 2 * kAccBufs + 1) * 8 + 4 <= 256, "mbarriers + TMEM slot fit 256 B");
static_assert(kNmax % kXBoxRows == 0 && kNmax <= 64, "token tile");

constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct TileInfo {
  int seg, m0, rows, nt;
};

// Items are (active expert, 128-row weight tile); an active expert owns exactly one m-tile here.
__device__ __forceinline__ TileInfo decode_item(int item, int n_tiles, const int32_t* s_tile,
                                                const int32_t* s_seg, int nseg) {
  TileInfo t;
  const int mt = item / n_tiles;
  t.nt = item - mt * n_tiles;
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tile[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  t.seg = lo;
  t.m0 = s_seg[lo];
  t.rows = min(kNmax, s_seg[lo + 1] - t.m0);
  return t;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* drain = acc_empty + kAccBufs;
  uint64_t* sf_done = drain + 1;   // a stage's scale factors are in tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_done + kStages);
  int32_t* s_tile = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + 256);
  int32_t* s_seg = s_tile + (p.nseg + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);  // the copy-issuing thread (expect_tx)
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(sf_done + s), 1);
    fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
  // plan_early: the plan was written two kernels back and is complete (the kernel in between
  // waited for it before it let this one start), so only the copy issuer waits, and only before
  // its first load of the previous kernel's output; the weights of the first stages are in
  // flight by then
  if (!p.plan_early) griddep_wait();
  griddep_launch();
  for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) {
    s_tile[i] = __ldcg(p.tile_start + i);
    s_seg[i] = __ldcg(p.seg_off + i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_tiles = p.N / 128;
  int total = s_tile[p.nseg] * n_tiles;
  if (total < 0 || total > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_INVALID_ARG);
    total = 0;
  }
  const int kst = p.K / kBK;
  const uint32_t smem0 = smem_u32(smem);

  if (warp == kTmaWarp) {
    // ---------------- all operands: bulk copies + one 2-D TMA tile per stage ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // only the boxes that hold the expert's rows (16 rows each); the rest of the token tile
      // stays stale and only feeds accumulator columns that are never stored
      auto stage_bytes = [&](const TileInfo& t) {
        return (uint32_t)(kTileBlockBytes + ((max(t.rows, 1) + kXBoxRows - 1) / kXBoxRows) *
                                                kXBoxRows * 128 + kXSfBytes);
      };
      // weight blocks of the first stages (the ring is empty: no wait), before the wait for
      // the previous kernel's output
      int pre = 0;
      if (p.plan_early) {
        for (int item = blockIdx.x; item < total && pre < kStages; item += gridDim.x) {
          const TileInfo t = decode_item(item, n_tiles, s_tile, s_seg, p.nseg);
          const uint8_t* src = p.b_tiles + (size_t)t.seg * p.b_per_seg +
                               (size_t)t.nt * kst * kTileBlockBytes;
          for (int ks = 0; ks < kst && pre < kStages; ++ks, ++pre) {
            const uint32_t fb = smem_u32(full + pre);
            mbar_arrive_expect_tx(fb, stage_bytes(t));
            bulk_load(smem0 + pre * kStageBytes, src + (size_t)ks * kTileBlockBytes,
                      kTileBlockBytes, fb);
          }
        }
        griddep_wait();
      }
      int g = 0;   // stages issued so far
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const TileInfo t = decode_item(item, n_tiles, s_tile, s_seg, p.nseg);
        const uint8_t* src = p.b_tiles + (size_t)t.seg * p.b_per_seg +
                             (size_t)t.nt * kst * kTileBlockBytes;
        const uint8_t* xsf = p.a_sf_tiles + (size_t)s_tile[t.seg] * (p.K / 64) * 512;
        const int nbox = (max(t.rows, 1) + kXBoxRows - 1) / kXBoxRows;
        for (int ks = 0; ks < kst; ++ks, ++g) {
          const uint32_t sb = smem0 + stage * kStageBytes;
          const uint32_t fb = smem_u32(full + stage);
          if (g >= pre) {
            if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(fb, stage_bytes(t));
            bulk_load(sb, src + (size_t)ks * kTileBlockBytes, kTileBlockBytes, fb);
          }
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(sb + kXOff + bx * kXBoxRows * 128, &tmap_x, ks * 128,
                        t.m0 + bx * kXBoxRows, fb);
          bulk_load(sb + kXSfOff, xsf + (size_t)ks * kXSfBytes, kXSfBytes, fb);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int i = 0; i < kStages && ok; ++i) {
        if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, p.status)) break;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue: D[weight row][token] ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase[kAccBufs] = {};
      // stage 0's operand descriptors; a stage (or a K step) further is an addition to the
      // 14-bit address field, which never carries (shared addresses stay below 256 KB)
      const uint64_t dA0 = smem_desc(smem0, 16, 1024, kLayoutSwizzle128B);
      const uint64_t dB0 = smem_desc(smem0 + kXOff, 16, 1024, kLayoutSwizzle128B);
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        const TileInfo t = decode_item(item, n_tiles, s_tile, s_seg, p.nseg);
        const int nmma = max(16, (t.rows + 15) & ~15);
        const uint32_t idesc = make_idesc(128, nmma);
        const int abuf = it % kAccBufs;
        if (!mbar_wait_bounded(smem_u32(acc_empty + abuf), acc_phase[abuf] ^ 1u, kWaitLimitNs,
                               p.status)) {
          ok = false;
          break;
        }
        acc_phase[abuf] ^= 1u;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * kAccCols;
        for (int ks = 0; ks < kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(sf_done + stage), phase, kWaitLimitNs, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((uint32_t)(stage * kStageBytes) >> 4);
          const uint32_t sf_t = tmem_base + kSfCol0 + stage * kSfColsPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // K = 64 per MMA: 32 bytes -> 2 descriptor units
            tc_mma_mxf4nvf4(d_tmem, dA0 + so + kk * 2, dB0 + so + kk * 2, idesc, sf_t + kk * 4,
                            sf_t + 16 + kk * 4, (ks | kk) != 0 ? 1u : 0u);
          tc_commit(smem_u32(empty + stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc_commit(smem_u32(acc_full + abuf));
      }
      tc_commit(smem_u32(drain));
      mbar_wait_bounded(smem_u32(drain), 0u, kWaitLimitNs, p.status);
    }
  } else if (warp == kSfWarp) {
    // ---------------- scale factors: shared -> tensor memory, ahead of the MMA thread ---------
    // A stage's scale columns are rewritten only after the copy engine refilled the stage, which
    // waited for the MMAs of its previous use to complete.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint64_t dSw0 = smem_desc(smem0 + kTileBytes, 0, 128, kLayoutSwizzleNone);
      const uint64_t dSx0 = smem_desc(smem0 + kXSfOff, 0, 128, kLayoutSwizzleNone);
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        for (int ks = 0; ks < kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(full + stage), phase, kWaitLimitNs, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((uint32_t)(stage * kStageBytes) >> 4);
          const uint32_t sf_t = tmem_base + kSfCol0 + stage * kSfColsPerStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {   // one 512-byte scale group per K = 64
            tc_cp_32x128b_warpx4(sf_t + kk * 4, dSw0 + so + kk * 32);
            tc_cp_32x128b_warpx4(sf_t + 16 + kk * 4, dSx0 + so + kk * 32);
          }
          tc_commit(smem_u32(sf_done + stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 0-3): lane = weight row, column = token ----------------
    uint32_t acc_phase[kAccBufs] = {};
    int it = 0;
    const float ts_a = p.mode == 0 ? *p.ts_a : 0.0f;
    const float inv_ts_h = 1.0f / p.ts_h;
    const bool lo_half = lane < 16;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      const TileInfo t = decode_item(item, n_tiles, s_tile, s_seg, p.nseg);
      const int abuf = it % kAccBufs;
      if (!mbar_wait_bounded(smem_u32(acc_full + abuf), acc_phase[abuf], kWaitLimitNs, p.status))
        break;
      acc_phase[abuf] ^= 1u;
      tc_fence_after();
      const int rows = (t.m0 >= 0 && t.m0 + t.rows <= p.out_rows) ? t.rows : 0;
      const uint32_t tbase = tmem_base + abuf * kAccCols + ((uint32_t)(warp * 32) << 16);
      if (p.mode == 0) {
        // block b of h: 16 features; lanes < 16 hold gate rows, lanes >= 16 the up rows
        const int I = p.N / 2;
        const int b = t.nt * 4 + warp;
        uint8_t* hsf_tile = p.hsf_tiles + ((size_t)s_tile[t.seg] * (I / 64) + b / 4) * 512 + (b & 3);
        const float ag = ts_a * p.w_ts[t.seg * 4 + 0];
        const float au = ts_a * p.w_ts[t.seg * 4 + 1];
#pragma unroll 1
        for (int cb = 0; cb < kNmax; cb += 32) {
          if (cb >= rows) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + cb, v);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < 32; n += 2) {
            if (cb + n >= rows) break;
            const float a0 = __uint_as_float(v[n]), a1 = __uint_as_float(v[n + 1]);
            const float x0 = __shfl_xor_sync(0xffffffffu, a0, 16);
            const float x1 = __shfl_xor_sync(0xffffffffu, a1, 16);
            // the lower half-warp takes token cb+n, the upper half token cb+n+1
            float g = (lo_half ? a0 : x1) * ag;
            float u = (lo_half ? x0 : a1) * au;
            const int col = cb + n + (lo_half ? 0 : 1);
            if (p.swiglu_clamp) {   // gate clamped from above, up on both sides
              g = fminf(g, p.swiglu_limit);
              u = fminf(fmaxf(u, -p.swiglu_limit), p.swiglu_limit);
            }
            const float h = silu_mul(g, u);
            float bamax = fabsf(h);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) bamax = fmaxf(bamax, __shfl_xor_sync(0xffffffffu, bamax, o));
            uint32_t sf = 0u;
            float q = 0.0f;
            if (bamax != 0.0f) {
              sf = f32_to_e4m3(bamax * (1.0f / 6.0f) * inv_ts_h);
              const float S = e4m3_to_f32(sf) * p.ts_h;
              if (S != 0.0f) q = h * __frcp_rn(S);
            }
            // gather the eight quotients of each quarter-warp into its first lane
            const int g0 = lane & ~7;
            float qq[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) qq[e] = __shfl_sync(0xffffffffu, q, g0 + e);
            const uint32_t word = e2m1x8(qq[0], qq[1], qq[2], qq[3], qq[4], qq[5], qq[6], qq[7]);
            const uint32_t word_hi = __shfl_down_sync(0xffffffffu, word, 8);
            if ((lane & 15) == 0 && col < rows) {
              const size_t prow = (size_t)(t.m0 + col);
              *reinterpret_cast<uint2*>(p.hq + prow * (I / 2) + b * 8) = make_uint2(word, word_hi);
              p.hsf[prow * (I / 16) + b] = (uint8_t)sf;
              hsf_tile[(col & 31) * 16 + (col >> 5) * 4] = (uint8_t)sf;
            }
          }
        }
      } else {
        // output features m = nt*128 + warp*32 + lane; token column n -> permuted row m0 + n
        const float alpha = p.ts_h * p.w_ts[t.seg * 4 + 2];
        const int m = t.nt * 128 + warp * 32 + lane;
        float wr[2] = {0.0f, 0.0f};
        int tok[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = lane + 32 * i;
          if (r < rows) {
            wr[i] = __ldg(p.perm_w + t.m0 + r);
            int tk = __ldg(p.perm_src + t.m0 + r);
            if (tk < 0 || tk >= p.y_rows) {
              set_status(p.status, MOE_ERR_INVALID_ARG);
              tk = -1;
            }
            tok[i] = tk;
          }
        }
#pragma unroll 1
        for (int cb = 0; cb < kNmax; cb += 32) {
          if (cb >= rows) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + cb, v);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            if (cb + n >= rows) break;
            const float w = __shfl_sync(0xffffffffu, wr[cb >> 5], n);
            const float d = (__uint_as_float(v[n]) * alpha) * w;
            if (p.mode == 2) {
              p.obuf[(size_t)(t.m0 + cb + n) * p.N + m] = d;
            } else {
              const int tk = __shfl_sync(0xffffffffu, tok[cb >> 5], n);
              if (tk >= 0) red_add_f32(p.yacc + (size_t)tk * p.N + m, d);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + abuf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t smem_bytes(int nseg) {
  return 1024 + (size_t)kStages * kStageBytes + 256 + sizeof(int32_t) * 2 * (nseg + 2);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

bool tensor_map_available() { return encode_fn() != nullptr; }

cudaError_t launch_grouped_gemm_decode(const GemmArgs& a, cudaStream_t s) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  // token rows [out_rows, K/2] bytes in expert order; box = 128 bytes x 16 rows, 128B swizzle
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 2), (cuuint64_t)a.out_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 2)};
  const cuuint32_t box[2] = {128, (cuuint32_t)kXBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.a_codes), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = smem_bytes(a.nseg);
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = a.max_ctas;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  return launch_pdl(grouped_gemm_decode_kernel, dim3(grid), dim3(kThreads), smem, s, tmap, a);
}

}  // namespace nvfp4moe
