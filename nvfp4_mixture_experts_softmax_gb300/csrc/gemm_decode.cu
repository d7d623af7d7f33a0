// Both grouped block-scaled FP4 GEMMs of a decode-sized batch (at most 64 tokens) in one
// persistent launch, with the operands swapped: the expert's weights are the MMA's A operand
// (M = 128 weight rows of one packed block per K stage, loaded by one bulk copy) and a tile of at
// most 16 of the expert's token rows is the B operand (N = 16; an expert with more rows owns
// several tiles).  The tensor core then works on the real tokens only, a pipeline stage is
// 22.5 KB (nine stages in flight), and the accumulator holds one weight row per TMEM lane and one
// token per column.
//   GEMM1 items (phase 0): warp w of the epilogue holds the 16 gate rows and the 16 up rows of
//          one 16-feature NVFP4 block, so each half-warp computes silu(g)*u of one token and
//          requantises the block with half-warp reductions; each warp then publishes its share
//          of the expert's h rows (release add on the expert's readiness count);
//   GEMM2 items (phase 1): lanes hold consecutive output features, so a token's router-weighted
//          row is stored 128 contiguous bytes per warp.
// Every CTA takes its GEMM1 items first, then its GEMM2 items, all through one ring of stages:
// one thread streams the weight blocks into every slot as soon as it is free (weights depend on
// nothing but the plan), another adds each stage's token rows once they exist - the activations
// after the prologue, the h rows of a GEMM2 item after all GEMM1 tiles of its expert are
// published - and a stage is full when both parts have landed.
// This removes the second launch's ramp and the full drain between the two GEMMs, which at
// decode sizes cost more than the weight stream itself.  CTAs wait on each other only through
// the readiness counts, and only after finishing every GEMM1 item of their own, so with one CTA
// per SM and a grid no larger than the SM count they cannot deadlock; every wait is bounded.
// Every operand arrives by the copy engine: per stage one bulk copy of the weight block, 2-D TMA
// tiles (128-byte swizzle) of the expert's token rows - the activations (GEMM1) or h (GEMM2) are
// stored in expert order, so an expert's rows are contiguous - and one bulk copy of the tokens'
// scales, which the producers write pre-arranged per expert tile.  Warps: 0-3 epilogue, 4 weight
// copies, 5 MMA, 6 scale factors, 7 token copies ("nvfp4-megamoe-kernel compare pre-b1...master",
// section "MoE kernel": TMA, MMA and epilogue warps; the pages keep decode on 1-CTA tiles).  The
// eight shared -> tensor memory scale copies of a stage hold up the thread that issues them for a long
// time, so a warp of their own issues them one stage ahead of the MMA thread and signals it
// through an mbarrier; the MMA thread then issues only the four MMAs of a stage, with
// descriptors advanced by additions.  Three TMEM accumulators let the epilogue trail the main
// loop by up to two tiles.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kStages = 9;
constexpr int kAccBufs = 3;
constexpr int kXBoxRows = 16;                          // token rows per TMA box
constexpr int kEpiWarps = 4;
constexpr int kWeightWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSfWarp = 6;
constexpr int kXWarp = 7;                              // token rows (and what they wait for)
constexpr int kThreads = (kXWarp + 1) * 32;
constexpr int kNmax = kDecodeTileRows;                // token rows per tile (the MMA N)
constexpr int kXOff = kTileBlockBytes;                 // token codes after the weight block
constexpr int kXBytes = kNmax * 128;
constexpr int kXSfOff = kXOff + kXBytes;               // token scales
constexpr int kXSfBytes = 4 * 512;
constexpr int kStageBytes = kXSfOff + kXSfBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 32;                      // accumulator spacing (>= kNmax)
constexpr uint32_t kSfCol0 = kAccBufs * kAccCols;
constexpr uint32_t kSfColsPerStage = 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kBarBytes = 512;                          // mbarriers + TMEM slot

static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(kStageBytes % 1024 == 0 && kXOff % 1024 == 0, "1024-byte aligned swizzled tiles");
constexpr size_t kMaxDynSmem = 232448;                   // 227 KB per CTA
// plan arrays of up to 1025 segments and a tile table of up to 2112 tiles (64 tokens, k <= 32,
// plus the shared expert's rows)
static_assert(kStages * kStageBytes + 1024 + kBarBytes + 4 * (2 * 1028 + 2112) <= kMaxDynSmem,
              "shared memory");
static_assert((3 * kStages + 2 * kAccBufs + 3) * 8 + 6 * 4 <= kBarBytes,
              "mbarriers, TMEM slot, issue counts and plan flags");
static_assert(kNmax == kXBoxRows && kNmax <= (int)kAccCols, "one TMA box of token rows per stage");

constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One work item: (m-tile, 128-row weight tile) of GEMM1 (phase 0, items [0, total1)) or of GEMM2
// (phase 1, items [total1, total1 + total2)).  An m-tile is kNmax consecutive rows of one expert
// (s_tseg gives its segment); an expert with more rows than that owns several.
struct Item {
  int ph, seg, mt, m0, rows, nt, kst;
};

__device__ __forceinline__ Item decode_item(int item, int total1, int nt1, int nt2, int kst1,
                                            int kst2, const int32_t* s_tseg, const int32_t* s_seg,
                                            const int32_t* s_tile) {
  Item t;
  t.ph = item >= total1 ? 1 : 0;
  const int local = t.ph ? item - total1 : item;
  const int ntl = t.ph ? nt2 : nt1;
  t.mt = local / ntl;
  t.nt = local - t.mt * ntl;
  t.kst = t.ph ? kst2 : kst1;
  t.seg = s_tseg[t.mt];    // always in [0, nseg): every entry is initialised
  t.m0 = s_seg[t.seg] + (t.mt - s_tile[t.seg]) * kNmax;
  t.rows = min(kNmax, s_seg[t.seg + 1] - t.m0);
  return t;
}

template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmap_x,
                               const __grid_constant__ CUtensorMap tmap_h,
                               const DecodeGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  // the 1024-byte-aligned base, reached by pointer arithmetic on the shared array so that the
  // compiler keeps the shared address space (shared loads and stores, not generic ones)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* drain = acc_empty + kAccBufs;
  uint64_t* sf_done = drain + 1;   // a stage's scale factors are in tensor memory
  uint64_t* plan_bar = sf_done + kStages;   // the bulk copy of the plan
  uint64_t* sf_drain = plan_bar + 1;         // the scale-factor warp's last tensor-memory copies
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
  // stage fills issued by the weight and the token issuers, whether the plan copy may still be
  // in flight, and whether the plan is usable (read by every role after the plan barrier)
  uint32_t* s_issued = tmem_slot + 1;
  uint32_t* s_plan_pending = s_issued + 2;
  uint32_t* s_plan_ok = s_plan_pending + 1;
  volatile uint32_t* s_abort = s_plan_ok + 1;   // set by any role whose bounded wait ran out
  const int nseg = p.g1.nseg;
  const int plan_ints = (nseg + 1 + 3) & ~3;    // 16-byte multiples for the bulk copies
  // m-tiles can outnumber segments (an expert with more than kNmax rows owns several): the
  // m-tile -> segment table has an entry for every tile the launch can hold
  const int max_tiles = p.g1.max_items / (p.g1.N / 128);
  int32_t* s_tile = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + kBarBytes);
  int32_t* s_seg = s_tile + plan_ints;
  int32_t* s_tseg = s_seg + plan_ints;     // m-tile -> segment, max_tiles entries
  int32_t* status = p.g1.status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch();   // the row sum may be scheduled; it waits for this grid to complete
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 2);  // the weight and the token issuers (expect_tx each)
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(sf_done + s), 1);
    mbar_init(smem_u32(plan_bar), 1);
    mbar_init(smem_u32(sf_drain), 1);
    s_issued[0] = s_issued[1] = 0u;
    *s_plan_pending = 0u;
    *s_plan_ok = 0u;
    *s_abort = 0u;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kWeightWarp) {
    // The plan (segment offsets and tile starts) is published by the decode prologue before it
    // encodes the activations: waiting for that flag instead of the prologue's completion lets
    // the weight stream start while the prologue still runs.  A wait that times out leaves an
    // empty plan (no items) and the status word set.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_h) : "memory");
    }
    int ok = 1;
    if (lane == 0) {
      uint64_t t0 = 0;
      for (uint32_t i = 0; ld_acquire_s32(p.plan_flag) == 0; ++i) {
        if ((i & 63u) == 63u) {
          const uint64_t now = global_timer_ns();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > kWaitLimitNs) {
            set_status(status, MOE_ERR_DEVICE_TIMEOUT);
            ok = 0;
            break;
          }
        }
      }
      if (ok) {
        // both arrays in one round trip: two bulk copies (16-byte multiples; the arrays are
        // allocated in 256-byte units, so the rounded-up tail stays inside them)
        fence_proxy_async_global();
        const uint32_t bytes = (uint32_t)((4 * (nseg + 1) + 15) & ~15);
        const uint32_t pb = smem_u32(plan_bar);
        mbar_arrive_expect_tx(pb, 2 * bytes);
        bulk_load(smem_u32(s_tile), p.g1.tile_start, bytes, pb);
        bulk_load(smem_u32(s_seg), p.g1.seg_off, bytes, pb);
        if (!mbar_wait_bounded(pb, 0u, kWaitLimitNs, status)) {
          ok = 0;
          *s_plan_pending = 1u;   // the copy may still land: drained before the CTA exits
        }
      }
      *s_plan_ok = (uint32_t)ok;
      if (!ok) *s_abort = 1u;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (ok) {
      for (int i = lane; i < max_tiles; i += 32) s_tseg[i] = 0;
      __syncwarp();
      for (int sg = lane; sg < nseg; sg += 32)
        for (int mt = max(s_tile[sg], 0); mt < s_tile[sg + 1] && mt < max_tiles; ++mt)
          s_tseg[mt] = sg;
    }
  }
  // every role reads the plan (or, after a timeout, runs no item) only after this barrier; the
  // weight warp's waits above are bounded, so the barrier is reached
  __syncthreads();

  const int nt1 = p.g1.N / 128, nt2 = p.g2.N / 128;
  const int kst1 = p.g1.K / kBK, kst2 = p.g2.K / kBK;
  const int mtiles = *s_plan_ok ? s_tile[nseg] : 0;
  int total1 = mtiles * nt1, total2 = mtiles * nt2;
  if (mtiles < 0 || mtiles > max_tiles || total1 > p.g1.max_items || total2 > p.g2.max_items) {
    if (threadIdx.x == 0) set_status(status, MOE_ERR_INVALID_ARG);
    total1 = total2 = 0;
  }
  const int total = total1 + total2;
  // an expert's h rows are complete once every epilogue warp of its GEMM1 tiles has published
  const int ready_target = nt1 * kEpiWarps;
  const uint32_t smem0 = smem_u32(smem);
#define NVFP4MOE_ITEM(i) decode_item((i), total1, nt1, nt2, kst1, kst2, s_tseg, s_seg, s_tile)

  if (warp == kWeightWarp) {
    // ---------------- weight blocks: one bulk copy per stage ----------------
    // Weights depend on nothing but the plan, so this thread only waits for free ring slots;
    // the stage's token rows come from the token issuer (warp kXWarp), and the stage's full
    // barrier completes once both parts have landed.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, n_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const Item t = NVFP4MOE_ITEM(item);
        const GemmArgs& q = t.ph ? p.g2 : p.g1;
        const uint8_t* src = q.b_tiles + (size_t)t.seg * q.b_per_seg +
                             (size_t)t.nt * t.kst * kTileBlockBytes;
        for (int ks = 0; ks < t.kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(full + stage);
          mbar_arrive_expect_tx(fb, kTileBlockBytes);
          bulk_load(smem0 + stage * kStageBytes, src + (size_t)ks * kTileBlockBytes,
                    kTileBlockBytes, fb);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // the MMAs of the last stages must finish before the CTA may exit
      for (int i = 0; i < kStages && ok; ++i) {
        if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, status)) {
          ok = false;
          break;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      s_issued[0] = n_issued;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp == kXWarp) {
    // ---------------- token rows: one 2-D TMA box + their scales per stage ----------------
    // GEMM1 reads the activations the prologue encoded (the dependency wait), GEMM2 the h rows
    // of the item's expert once every GEMM1 epilogue warp of it has published them.
    if (lane == 0) {
      griddep_wait();
      int stage = 0;
      uint32_t phase = 0, n_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const Item t = NVFP4MOE_ITEM(item);
        const GemmArgs& q = t.ph ? p.g2 : p.g1;
        if (t.ph == 1) {
          uint64_t t0 = 0;
          for (uint32_t i = 0; ld_acquire_s32(p.ready + t.mt) < ready_target; ++i) {
            if ((i & 63u) == 63u) {
              const uint64_t now = global_timer_ns();
              if (t0 == 0) {
                t0 = now;
              } else if (now - t0 > kWaitLimitNs) {
                set_status(status, MOE_ERR_DEVICE_TIMEOUT);
                ok = false;
                break;
              }
            }
          }
          if (!ok) break;
          fence_proxy_async_global();
        }
        const void* tm = t.ph ? (const void*)&tmap_h : (const void*)&tmap_x;
        const uint8_t* sft = q.a_sf_tiles + (size_t)t.mt * (q.K / 64) * 512;
        const uint32_t xbytes = (uint32_t)(kXBoxRows * 128 + kXSfBytes);
        for (int ks = 0; ks < t.kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, kWaitLimitNs, status)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem0 + stage * kStageBytes;
          const uint32_t fb = smem_u32(full + stage);
          mbar_arrive_expect_tx(fb, xbytes);
          tma_load_2d(sb + kXOff, tm, ks * 128, t.m0, fb);
          bulk_load(sb + kXSfOff, sft + (size_t)ks * kXSfBytes, kXSfBytes, fb);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      s_issued[1] = n_issued;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue: D[weight row][token] ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
      // stage 0's operand descriptors; a stage (or a K step) further is an addition to the
      // 14-bit address field, which never carries (shared addresses stay below 256 KB)
      const uint64_t dA0 = smem_desc(smem0, 16, 1024, kLayoutSwizzle128B);
      const uint64_t dB0 = smem_desc(smem0 + kXOff, 16, 1024, kLayoutSwizzle128B);
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        const Item t = NVFP4MOE_ITEM(item);
        const int nmma = max(16, (t.rows + 15) & ~15);
        const uint32_t idesc = make_idesc(128, nmma);
        const int abuf = it % kAccBufs;
        const uint32_t acc_par = (acc_phase >> abuf) & 1u;
        if (!mbar_wait_bounded(smem_u32(acc_empty + abuf), acc_par ^ 1u, kWaitLimitNs,
                               status)) {
          ok = false;
          break;
        }
        acc_phase ^= 1u << abuf;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * kAccCols;
        for (int ks = 0; ks < t.kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(sf_done + stage), phase, kWaitLimitNs, status)) {
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
      if (!mbar_wait_bounded(smem_u32(drain), 0u, kWaitLimitNs, status)) ok = false;
      if (!ok) *s_abort = 1u;
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
        const int kst = item < total1 ? kst1 : kst2;
        for (int ks = 0; ks < kst; ++ks) {
          if (!mbar_wait_bounded(smem_u32(full + stage), phase, kWaitLimitNs, status)) {
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
      if (!ok) *s_abort = 1u;
    }
  } else {
    // ---------------- epilogue (warps 0-3): lane = weight row, column = token ----------------
    griddep_wait();     // the activation tensor scale and the router weights
    uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
    int it = 0;
    const float ts_a = *p.g1.ts_a;
    const float ts_h = p.g1.ts_h;
    const float inv_ts_h = 1.0f / ts_h;
    const bool lo_half = lane < 16;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      const Item t = NVFP4MOE_ITEM(item);
      const GemmArgs& q = t.ph ? p.g2 : p.g1;
      const int abuf = it % kAccBufs;
      // every lane waits; the decision is taken together so that the warp never diverges
      // before the warp-wide tensor-memory loads
      const uint32_t acc_par = (acc_phase >> abuf) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_full + abuf), acc_par,
                                                     kWaitLimitNs, status))) {
        if (lane == 0) *s_abort = 1u;
        break;
      }
      acc_phase ^= 1u << abuf;
      tc_fence_after();
      const int rows = (t.m0 >= 0 && t.m0 + t.rows <= q.out_rows) ? t.rows : 0;
      const uint32_t tbase = tmem_base + abuf * kAccCols + ((uint32_t)(warp * 32) << 16);
      if (t.ph == 0) {
        // Gated experts: block b of h (16 features); lanes < 16 hold its gate rows, lanes >= 16
        // its up rows, and each half-warp takes one token of a pair.  Non-gated experts (ReLU2):
        // lanes < 16 hold the up rows of block 2w, lanes >= 16 those of block 2w + 1 (w = the
        // warp's 32-row slice of the tile), and both halves take the same token.
        constexpr bool gated = kGated;
        const int I = gated ? q.N / 2 : q.N;
        const int b = gated ? t.nt * 4 + warp : t.nt * 8 + warp * 2 + (lo_half ? 0 : 1);
        uint8_t* hsf_tile = q.hsf_tiles + ((size_t)t.mt * (I / 64) + b / 4) * 512 + (b & 3);
        const float ag = ts_a * q.w_ts[t.seg * 4 + 0];
        const float au = ts_a * q.w_ts[t.seg * 4 + 1];
        if (rows > 0) {
          uint32_t v[kNmax];
          tmem_ld_32x32b_x16(tbase, v);
          tmem_ld_wait();
          // h of one token column per half-warp -> its NVFP4 block (half-warp reductions), codes
          // and scale stored by the half's first lane
          auto requant_store = [&](float h, int col) {
            float bamax = fabsf(h);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) bamax = fmaxf(bamax, __shfl_xor_sync(0xffffffffu, bamax, o));
            uint32_t sf = 0u;
            float qv = 0.0f;
            if (bamax != 0.0f) {
              sf = f32_to_e4m3(bamax * (1.0f / 6.0f) * inv_ts_h);
              const float S = e4m3_to_f32(sf) * ts_h;
              if (S != 0.0f) qv = h * __frcp_rn(S);
            }
            // gather the eight quotients of each quarter-warp into its first lane
            const int g0 = lane & ~7;
            float qq[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) qq[e] = __shfl_sync(0xffffffffu, qv, g0 + e);
            const uint32_t word = e2m1x8(qq[0], qq[1], qq[2], qq[3], qq[4], qq[5], qq[6], qq[7]);
            const uint32_t word_hi = __shfl_down_sync(0xffffffffu, word, 8);
            if ((lane & 15) == 0 && col < rows) {
              const size_t prow = (size_t)(t.m0 + col);
              *reinterpret_cast<uint2*>(q.hq + prow * (I / 2) + b * 8) = make_uint2(word, word_hi);
              q.hsf[prow * (I / 16) + b] = (uint8_t)sf;
              hsf_tile[col * 16] = (uint8_t)sf;
            }
          };
          if constexpr (kGated) {
#pragma unroll
            for (int n = 0; n < kNmax; n += 2) {
              if (n >= rows) break;
              const float a0 = __uint_as_float(v[n]), a1 = __uint_as_float(v[n + 1]);
              const float x0 = __shfl_xor_sync(0xffffffffu, a0, 16);
              const float x1 = __shfl_xor_sync(0xffffffffu, a1, 16);
              // the lower half-warp takes token n, the upper half token n+1
              const float g = (lo_half ? a0 : x1) * ag;
              const float u = (lo_half ? x0 : a1) * au;
              requant_store(glu_activation(g, u, q.act, q.swiglu_limit, q.swiglu_alpha),
                            n + (lo_half ? 0 : 1));
            }
          } else {
#pragma unroll
            for (int n = 0; n < kNmax; ++n) {
              if (n >= rows) break;
              requant_store(glu_activation(0.0f, __uint_as_float(v[n]) * au, q.act,
                                           q.swiglu_limit, q.swiglu_alpha),
                            n);
            }
          }
        }
      } else {
        // output features m = nt*128 + warp*32 + lane; token column n -> permuted row m0 + n
        const float alpha = ts_h * q.w_ts[t.seg * 4 + 2];
        const int m = t.nt * 128 + warp * 32 + lane;
        const float wr = lane < rows ? __ldg(q.perm_w + t.m0 + lane) : 0.0f;
        if (rows > 0) {
          uint32_t v[kNmax];
          tmem_ld_32x32b_x16(tbase, v);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < kNmax; ++n) {
            if (n >= rows) break;
            const float w = __shfl_sync(0xffffffffu, wr, n);
            q.obuf[(size_t)(t.m0 + n) * q.N + m] = (__uint_as_float(v[n]) * alpha) * w;
          }
        }
      }
      // the accumulator is free once its values are in registers; the publication of h below
      // waits for this warp's stores and stays off the MMA thread's path
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + abuf));
      if (t.ph == 0) {
        // publish this warp's share of the expert's h rows to the copy engines of every CTA
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add_s32(p.ready + t.mt, 1);
      }
    }
  }
#undef NVFP4MOE_ITEM

  // Teardown.  After a wait ran out, copies into shared memory may still be in flight: a stage
  // whose fill one issuer made and the other did not gets the missing arrival here (the leading
  // issuer is at most kStages fills ahead, since every fill waits for the slot's release, which
  // needs the previous phase complete), so every issued phase completes once its bytes land;
  // then the last kStages fills, the plan copy and the scale-factor thread's last tensor-memory
  // copies are waited for (bounded) before tensor memory is released.  Without a timeout every
  // fill and copy was consumed by a completed MMA, and none of this runs.
  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    if (warp == kWeightWarp && lane == 0) {
      const uint32_t wi = s_issued[0], xi = s_issued[1];
      const uint32_t lo = min(wi, xi), hi = max(wi, xi);
      for (uint32_t i = lo; i < hi; ++i) mbar_arrive(smem_u32(full + i % kStages));
      for (uint32_t i = hi > (uint32_t)kStages ? hi - kStages : 0u; i < hi; ++i)
        if (!mbar_wait_bounded(smem_u32(full + i % kStages), (i / kStages) & 1u, kWaitLimitNs,
                               status))
          break;
      if (*s_plan_pending) mbar_wait_bounded(smem_u32(plan_bar), 0u, kWaitLimitNs, status);
    } else if (warp == kSfWarp && lane == 0) {
      tc_commit(smem_u32(sf_drain));
      mbar_wait_bounded(smem_u32(sf_drain), 0u, kWaitLimitNs, status);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t smem_bytes(int nseg, int max_tiles) {
  return 1024 + (size_t)kStages * kStageBytes + kBarBytes +
         sizeof(int32_t) * (2 * ((nseg + 1 + 3) & ~3) + (size_t)max_tiles);
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

namespace {

// Token rows [rows, K/2] bytes in expert order; box = 128 bytes x 16 rows, 128-byte swizzle.
bool encode_token_map(CUtensorMap* tmap, const uint8_t* codes, int K, int rows) {
  auto encode = encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {128, (cuuint32_t)kXBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_gemm_decode(const DecodeGemmArgs& a, cudaStream_t s) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.g1.nseg != a.g2.nseg || a.g1.tile_start != a.g2.tile_start || a.g1.seg_off != a.g2.seg_off ||
      a.g1.mode != 0 || a.g2.mode != 2 || !a.ready || !a.plan_flag)
    return cudaErrorInvalidValue;
  CUtensorMap tmap_x, tmap_h;
  if (!encode_token_map(&tmap_x, a.g1.a_codes, a.g1.K, a.g1.out_rows) ||
      !encode_token_map(&tmap_h, a.g2.a_codes, a.g2.K, a.g2.out_rows))
    return cudaErrorInvalidValue;
  const int nt1 = a.g1.N / 128;
  if (nt1 < 1 || a.g1.max_items % nt1 != 0) return cudaErrorInvalidValue;
  const size_t smem = smem_bytes(a.g1.nseg, a.g1.max_items / nt1);
  if (smem > kMaxDynSmem) return cudaErrorInvalidValue;
  // one instantiation per GEMM1 layout (gate/up interleaved, or up rows alone), so that the
  // epilogue of either carries no code for the other
  auto kernel = a.g1.act == kActRelu2 ? grouped_gemm_decode_kernel<false>
                                      : grouped_gemm_decode_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM at most: CTAs wait on each other's GEMM1 tiles, so all of them must be
  // resident together (one 200 KB CTA fits an SM; the grid never exceeds the SM count)
  const int64_t items = (int64_t)a.g1.max_items + a.g2.max_items;
  int grid = (int)std::min<int64_t>(items, num_sms());
  if (grid < 1) grid = 1;
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, tmap_x, tmap_h, a);
}

}  // namespace nvfp4moe
