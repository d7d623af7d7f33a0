// Persistent grouped GEMM on the 5th-generation tensor cores with block-scaled FP4 operands
// (tcgen05.mma kind::mxf4nvf4, E2M1 values, one E4M3 scale per 16 elements), used twice per layer
// for batches larger than the decode path's:
//   GEMM1: the expert-ordered quantised activations x the expert's interleaved gate/up weights
//          (or up weights alone for non-gated experts); the epilogue applies the tensor scales,
//          the activation (SwiGLU silu(g)*u, clamped, gpt-oss, or ReLU2), and requantises h to NVFP4
//          ("nvfp4-megamoe-kernel compare pre-b1...master", section "MoE kernel
//          (FusedSwiGLUScaledGroupedGemmKernel)": epilogue with global scale + SwiGLU in
//          registers between the tensor-memory load and the store);
//   GEMM2: h x the expert's down weights; the epilogue scales by the tensor scales and the router
//          weight and reduces into the token's FP32 output row (or stores the row)
//          ("vllm.cpp docs/STATUS.md", row "Brick C part 1": y = sum_j w_j * expert_out_j).
//
// Tiles are 128 expert-ordered rows (MMA M) x 128 weight rows (MMA N), K in stages of 256.  Every
// operand arrives by the copy engine: per stage one 2-D TMA box of the 128 activation rows
// (128-byte swizzle; an expert's rows are contiguous in the expert-ordered buffer), one bulk
// copy of their pre-arranged scales, and one bulk copy of the packed weight block.  One CTA per
// SM, warp-specialised (the pages' design uses TMA / MMA / epilogue warps and a scheduler warp;
// here the schedule is a static round robin over the device-built tile list):
//   warps 0-3  epilogue: tensor memory -> registers -> global, one accumulator row per thread;
//   warp  4    copy issue; warp 5 tensor-memory allocation and the single MMA-issuing thread;
//   warp  6    the eight shared -> tensor memory scale-factor copies of each stage, one stage
//              ahead of the MMA thread (issued from the MMA thread they stall it for long
//              enough to starve the tensor core).
// A 6-stage shared-memory ring (5 stages for the reducing epilogue, whose transpose buffers take
// the rest) of mbarrier full/empty pairs feeds the MMA; two 128-column FP32 accumulators let the
// epilogue of one tile overlap the main loop of the next.  Every wait is
// bounded in time and reports MOE_ERR_DEVICE_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kEpiWarps = 4;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSfWarp = 6;
constexpr int kThreads = (kSfWarp + 1) * 32;
// Stage layout: A codes | A scales | B block (codes + scales, one packed weight block).
constexpr int kABytes = kBM * 128;
constexpr int kSfBytes = 4 * 512;  // four 512-byte scale groups (one per 64-wide MMA K step)
constexpr int kBOff = kABytes + kSfBytes;
constexpr int kStageBytes = kBOff + kTileBlockBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kBN;
constexpr uint32_t kSfCol0 = 2 * kAccCols;
constexpr uint32_t kSfColsPerStage = 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kBN == 128 && kTileBlockBytes == kBN * 128 + kSfBytes, "packed block = B stage");
static_assert(kBOff % 1024 == 0, "B tile stays 1024-byte aligned for the 128B swizzle");
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");

// The reducing epilogue (mode 1) adds router-weighted FP32 rows into the L2-resident token
// accumulator in one of two ways:
//  kRed == 1: each warp's 32 x 32 chunk is transposed through shared memory so that one vector
//    reduction instruction covers four rows x 128 contiguous bytes (eight lanes per row).
//    16-byte unit q of row r sits at r * 128 + ((q ^ (r & 7)) * 16): conflict free both ways.
//    4 KB per warp.
//  kRed == 2: each lane's whole 128-column row goes to shared memory and then to the bulk-copy
//    engine as one 512-byte reduce-add, performed by the memory system; rows sit 528 bytes apart
//    so the eight lanes of a 16-byte store phase cover all 32 banks.  16.5 KB per warp.
// The second frees the epilogue warps sooner (one instruction per row instead of 32) but its
// rows cost the ring a stage; it wins when an item has few K stages (the epilogue dominates).
constexpr int kRedRowStride = kBN * 4 + 16;
template <int kRed>
constexpr int stg_buf_bytes() { return kRed == 2 ? 32 * kRedRowStride : kRed == 1 ? 32 * 128 : 0; }

// Ring depth: 6 stages for the SwiGLU / row-store epilogues, 5 with the transpose buffers, 4 with
// the bulk-reduction rows.
template <int kRed>
struct GemmShape {
  static constexpr int kStages = kRed == 2 ? 4 : kRed == 1 ? 5 : 6;
  static constexpr int kStgBufBytes = stg_buf_bytes<kRed>();
  static constexpr int kStgOff = kStages * kStageBytes;
  static constexpr int kBarOff = kStgOff + kEpiWarps * kStgBufBytes;
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
  static_assert(kBarOff + 1024 + 256 + 8 * 1027 <= 232448, "shared memory");
  // full, empty, sf_done per stage; two acc_full, two acc_empty, drain, sf_drain; TMEM slot and
  // the issue count, all before the plan arrays at kBarOff + 256
  static_assert((3 * kStages + 6) * 8 + 3 * 4 <= 256, "mbarriers + TMEM slot + counts");
};

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: A and B E2M1 (format 1) at bits 7-9 and
// 10-12, both K-major, N >> 3 at bits 17-22, UE4M3 scale type (bit 23 = 0), M >> 4 at bits 24-28,
// scale-factor ids 0, dense K = 64.
constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct TileInfo {
  int seg, m0, rows, nt;
};

__device__ __forceinline__ TileInfo decode_tile(int item, int n_tiles, const int32_t* s_tile,
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
  t.m0 = s_seg[lo] + (mt - s_tile[lo]) * kBM;
  t.rows = min(kBM, s_seg[lo + 1] - t.m0);
  return t;
}

template <int kRed>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  constexpr int kStages = GemmShape<kRed>::kStages;
  extern __shared__ uint8_t smem_raw[];
  // the 1024-byte-aligned base, reached by pointer arithmetic on the shared array so that the
  // compiler keeps the shared address space (shared loads and stores, not generic ones)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GemmShape<kRed>::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sf_done = drain + 1;   // a stage's scale factors are in tensor memory
  uint64_t* sf_drain = sf_done + kStages;   // the scale-factor warp's last tensor-memory copies
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
  uint32_t* s_issued = tmem_slot + 1;       // stage fills the copy thread issued
  volatile uint32_t* s_abort = s_issued + 1;   // set by any role whose bounded wait ran out
  int32_t* s_tile = reinterpret_cast<int32_t*>(smem + GemmShape<kRed>::kBarOff + 256);
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(sf_done + s), 1);
    mbar_init(smem_u32(sf_drain), 1);
    *s_issued = 0u;
    *s_abort = 0u;
    fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_a) : "memory");
  // everything above touched only shared and tensor memory; wait for the producer kernel now
  griddep_wait();
  griddep_launch();
  for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) {
    s_tile[i] = p.tile_start[i];
    s_seg[i] = p.seg_off[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_tiles = p.N / kBN;
  int total = s_tile[p.nseg] * n_tiles;
  if (total < 0 || total > p.max_items) {  // malformed plan: do nothing, report it
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_INVALID_ARG);
    total = 0;
  }
  const int kst = p.K / kBK;
  const uint32_t smem0 = smem_u32(smem);

  if (warp == kTmaWarp) {
    // ---------------- all operands: TMA box of A rows + bulk copies ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, n_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const TileInfo t = decode_tile(item, n_tiles, s_tile, s_seg, p.nseg);
        const uint8_t* bsrc = p.b_tiles + (size_t)t.seg * p.b_per_seg +
                              (size_t)t.nt * kst * kTileBlockBytes;
        // the global m-tile index is also the tile of the pre-arranged activation scales
        const uint8_t* asf = p.a_sf_tiles + (size_t)(item / n_tiles) * (p.K / 64) * 512;
        for (int ks = 0; ks < kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem0 + stage * kStageBytes;
          const uint32_t fb = smem_u32(full + stage);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d(sb, &tmap_a, ks * 128, t.m0, fb);
          bulk_load(sb + kABytes, asf + (size_t)ks * kSfBytes, kSfBytes, fb);
          bulk_load(sb + kBOff, bsrc + (size_t)ks * kTileBlockBytes, kTileBlockBytes, fb);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // tail: wait until the MMA has released every stage, so no arrival is still in flight
      for (int i = 0; i < kStages && ok; ++i) {
        if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, p.status)) {
          ok = false;
          break;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      *s_issued = n_issued;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
      // stage 0's operand descriptors; a stage (or a K step) further is an addition to the
      // 14-bit address field, which never carries (shared addresses stay below 256 KB)
      const uint64_t dA0 = smem_desc(smem0, 16, 1024, kLayoutSwizzle128B);
      const uint64_t dB0 = smem_desc(smem0 + kBOff, 16, 1024, kLayoutSwizzle128B);
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        const int abuf = it & 1;
        const uint32_t acc_par = (acc_phase >> abuf) & 1u;
        if (!mbar_wait_bounded(smem_u32(acc_empty + abuf), acc_par ^ 1u, kWaitLimitNs,
                               p.status)) {
          ok = false;
          break;
        }
        acc_phase ^= 1u << abuf;
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
      // make sure no tensor-core operation is still running before tensor memory is released
      tc_commit(smem_u32(drain));
      if (!mbar_wait_bounded(smem_u32(drain), 0u, kWaitLimitNs, p.status)) ok = false;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp == kSfWarp) {
    // ---------------- scale factors: shared -> tensor memory, ahead of the MMA thread ---------
    // A stage's scale columns are rewritten only after the copy engine refilled the stage, which
    // waited for the MMAs of its previous use to complete.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint64_t dSa0 = smem_desc(smem0 + kABytes, 0, 128, kLayoutSwizzleNone);
      const uint64_t dSb0 = smem_desc(smem0 + kBOff + kTileBytes, 0, 128, kLayoutSwizzleNone);
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
            tc_cp_32x128b_warpx4(sf_t + kk * 4, dSa0 + so + kk * 32);
            tc_cp_32x128b_warpx4(sf_t + 16 + kk * 4, dSb0 + so + kk * 32);
          }
          tc_commit(smem_u32(sf_done + stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) *s_abort = 1u;
    }
  } else {
    // ---------------- epilogue (warps 0-3) ----------------
    uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
    int it = 0;
    const int r = warp * 32 + lane;   // this thread's accumulator lane = tile row
    const float ts_a = p.mode == 0 ? *p.ts_a : 0.0f;
    const float inv_ts_h = 1.0f / p.ts_h;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      const TileInfo t = decode_tile(item, n_tiles, s_tile, s_seg, p.nseg);
      const int abuf = it & 1;
      // every lane waits; the decision is taken together so that the warp never diverges
      // before the warp-wide tensor-memory loads
      const uint32_t acc_par = (acc_phase >> abuf) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_full + abuf), acc_par,
                                                     kWaitLimitNs, p.status))) {
        if (lane == 0) *s_abort = 1u;
        break;
      }
      acc_phase ^= 1u << abuf;
      tc_fence_after();
      const int prow = t.m0 + r;
      const bool valid = r < t.rows && prow >= 0 && prow < p.out_rows;
      const uint32_t tbase = tmem_base + abuf * kAccCols + ((uint32_t)(warp * 32) << 16);
      if (p.mode == 0) {
        const float ag = ts_a * p.w_ts[t.seg * 4 + 0];
        const float au = ts_a * p.w_ts[t.seg * 4 + 1];
        const bool gated = p.act != kActRelu2;
        const int I = gated ? p.N / 2 : p.N;
        const size_t mt = (size_t)(item / n_tiles);
        const int rr = r & 127;
        uint8_t* hsf_tile = p.hsf_tiles + mt * (I / 64) * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, v);
          tmem_ld_wait();
          if (!valid) continue;
          // a 32-column chunk is one 16-feature block of h from (16 gate | 16 up) columns, or,
          // without a gate, two blocks from 32 up columns (indices stay compile-time constants so
          // that v stays in registers)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (gated && half == 1) break;
            float h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g = gated ? __uint_as_float(v[i]) * ag : 0.0f;
              const float u = __uint_as_float(gated ? v[16 + i] : v[16 * half + i]) * au;
              h[i] = glu_activation(g, u, p.act, p.swiglu_limit, p.swiglu_alpha);
            }
            uint32_t lo, hi, s;
            quant_block16_fast(h, p.ts_h, inv_ts_h, lo, hi, s);
            const int f0 = gated ? t.nt * (kBN / 2) + c * 16 : t.nt * kBN + c * 32 + half * 16;
            *reinterpret_cast<uint2*>(p.hq + (size_t)prow * (I / 2) + f0 / 2) = make_uint2(lo, hi);
            p.hsf[(size_t)prow * (I / 16) + f0 / 16] = (uint8_t)s;
            hsf_tile[(size_t)(f0 / 64) * 512 + ((f0 / 16) & 3)] = (uint8_t)s;
          }
        }
      } else {
        const float alpha = p.ts_h * p.w_ts[t.seg * 4 + 2];
        int tok = 0;
        float wr = 0.0f;
        bool ok_row = valid;
        if (valid) {
          tok = __ldg(p.perm_src + prow);
          wr = __ldg(p.perm_w + prow);
          if (tok < 0 || tok >= p.y_rows) {
            set_status(p.status, MOE_ERR_INVALID_ARG);
            ok_row = false;
            tok = 0;
          }
        }
        if constexpr (kRed == 2) {
          const uint32_t srow = smem0 + GemmShape<kRed>::kStgOff +
                                (uint32_t)warp * GemmShape<kRed>::kStgBufBytes +
                                (uint32_t)lane * kRedRowStride;
          bulk_wait_group_read<0>();   // this lane's previous reduction has read its row
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                               srow + (uint32_t)(c * 128 + i * 16)),
                           "f"((__uint_as_float(v[4 * i]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 1]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 2]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 3]) * alpha) * wr)
                           : "memory");
          }
          if (ok_row) {
            fence_proxy_async_smem();   // the row's stores, before the bulk engine reads them
            bulk_reduce_add_f32(p.yacc + (size_t)tok * p.N + t.nt * kBN, srow, kBN * 4);
            bulk_commit_group();
          }
        } else if constexpr (kRed == 1) {
          const uint32_t stg = smem0 + GemmShape<kRed>::kStgOff +
                               (uint32_t)warp * GemmShape<kRed>::kStgBufBytes;
          const uint32_t wrow = stg + (uint32_t)lane * 128;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                               wrow + (uint32_t)((i ^ (lane & 7)) * 16)),
                           "f"((__uint_as_float(v[4 * i]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 1]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 2]) * alpha) * wr),
                           "f"((__uint_as_float(v[4 * i + 3]) * alpha) * wr)
                           : "memory");
            __syncwarp();
            // lane l adds 16 bytes (unit l % 8) of row 4 * j + l / 8
            const int q = lane & 7;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int rj = 4 * j + (lane >> 3);
              const int ok_j = __shfl_sync(0xffffffffu, (int)ok_row, rj);
              const int tok_j = __shfl_sync(0xffffffffu, tok, rj);
              float4 d;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(d.x), "=f"(d.y), "=f"(d.z), "=f"(d.w)
                           : "r"(stg + (uint32_t)rj * 128 + (uint32_t)((q ^ (rj & 7)) * 16)));
              if (ok_j)
                red_add_v4(p.yacc + (size_t)tok_j * p.N + t.nt * kBN + c * 32 + 4 * q, d.x, d.y,
                           d.z, d.w);
            }
            __syncwarp();
          }
        } else {
          float* yrow = p.obuf + (size_t)(ok_row ? prow : 0) * p.N + t.nt * kBN;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
            if (ok_row) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(yrow + c * 32 + 4 * i) =
                    make_float4((__uint_as_float(v[4 * i]) * alpha) * wr,
                                (__uint_as_float(v[4 * i + 1]) * alpha) * wr,
                                (__uint_as_float(v[4 * i + 2]) * alpha) * wr,
                                (__uint_as_float(v[4 * i + 3]) * alpha) * wr);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + abuf));
    }
  }

  // Teardown.  After a wait ran out, stage fills and scale copies may still be in flight: the
  // copy thread's last kStages fills and the scale-factor thread's last tensor-memory copies are
  // waited for (bounded) before tensor memory is released.  Without a timeout every fill and
  // copy was consumed by a completed MMA, and none of this runs.  The reducing epilogue first
  // waits for its row reductions, whose sources live in shared memory.
  if constexpr (kRed == 2)
    if (warp < kEpiWarps) bulk_wait_group<0>();
  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    if (warp == kTmaWarp && lane == 0) {
      const uint32_t n = *s_issued;
      for (uint32_t i = n > (uint32_t)kStages ? n - kStages : 0u; i < n; ++i)
        if (!mbar_wait_bounded(smem_u32(full + i % kStages), (i / kStages) & 1u, kWaitLimitNs,
                               p.status))
          break;
    } else if (warp == kSfWarp && lane == 0) {
      tc_commit(smem_u32(sf_drain));
      mbar_wait_bounded(smem_u32(sf_drain), 0u, kWaitLimitNs, p.status);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int kRed>
size_t gemm_smem_bytes(int nseg) {
  return 1024 + (size_t)GemmShape<kRed>::kBarOff + 256 + sizeof(int32_t) * 2 * (nseg + 2);
}

template <int kRed>
cudaError_t launch_kernel(const CUtensorMap& tmap, const GemmArgs& a, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes<kRed>(a.nseg);
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kRed>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = a.max_ctas;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  return launch_pdl(grouped_gemm_kernel<kRed>, dim3(grid), dim3(kThreads), smem, s, tmap, a);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_general() {
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

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s) {
  auto encode = encode_fn_general();
  if (!encode) return cudaErrorNotSupported;
  // expert-ordered activation rows [out_rows, K/2] bytes; box = 128 bytes x 128 rows, 128B swizzle
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 2), (cuuint64_t)a.out_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 2)};
  const cuuint32_t box[2] = {128, (cuuint32_t)kBM};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.a_codes), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // reductions: bulk rows when an item has at most four K stages (measured: prefill GEMM2, K=512,
  // 217 -> 154 us), the transposed vector reductions and their deeper ring otherwise (K=1536 and
  // 2048 were 2-6% slower with bulk rows)
  if (a.mode != 1) return launch_kernel<0>(tmap, a, s);
  return a.K <= 4 * kBK ? launch_kernel<2>(tmap, a, s) : launch_kernel<1>(tmap, a, s);
}

}  // namespace nvfp4moe
