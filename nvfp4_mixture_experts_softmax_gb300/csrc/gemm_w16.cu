// Grouped GEMMs of the W4A16 layer: BF16 activations as they are, NVFP4 expert weights decoded
// to BF16 inside the kernel ("b12x" README, section "What's in here", moe: "W4A16 (BF16
// activations, inline FP4 weight dequant - no activation-scale math)"); and of the W4A8 layer
// (same page, "DeepSeek V4 Flash 0731 MoE reproduction": MXFP4 weights with one E8M0 scale per 32,
// MXFP8 activations), whose MXFP8 activations arrive already decoded to BF16 (exact), whose
// MXFP4 weights are decoded the same way as the NVFP4 ones (e2m1 * 2^(scale - 127), exact in
// BF16), and whose GEMM1 epilogue requantises h to MXFP8 (codes and scales are written out, the
// decoded BF16 values feed the down projection).  Exact decoding keeps the layer's arithmetic
// that of its definition: every product of two decoded operands is exact in FP32.
//
// Tiles are 256 expert-ordered token rows x 128 weight rows on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, BF16 x BF16 -> FP32 in tensor memory): each decoded weight tile is the
// N = 128 operand of two M = 128 MMAs, one per 128-row half of the token tile, K in sub-stages of
// 64.  Per K block of 256 the copy warp fetches the expert's packed NVFP4 weight block (18 KB,
// the layout the FP4 GEMMs read) with one bulk copy into a raw ring, and per sub-stage one 2-D
// TMA box (64 BF16 x 256 rows, 128-byte swizzle) of the expert-ordered activation rows.  The
// converter warps decode the sub-stage's 64 E2M1 codes of each weight row with their block
// scales into BF16 (e2m1 * scale has at most 6 significant bits and lies in [2^-10, 2688], so it
// is exact in BF16) by placing the codes' bits into BF16 fields and exact BF16 multiplications,
// with no per-element float conversion, and store the row into the sub-stage's weight tile in the
// same 128-byte-swizzled K-major layout; the per-matrix FP32 tensor scale is applied in the
// epilogue.  Batches of at most 64 tokens swap the operands: the decoded weight tile is the MMA's
// M = 128 and tiles of 16 expert-ordered token rows its N, so neither the MMA nor the token copies
// carry the padding of a large token tile (an active expert averages a few rows there); the
// epilogue then holds one weight row per thread and one token per accumulator column.
// Warps: 0-3 epilogue, 4 copies, 5 tensor-memory allocation + the MMA thread, 6-13 converters
// (two per weight row, each decoding half of the sub-stage's 64 codes: two converter warps per
// scheduler hide the decode's dependent instruction chains; with one warp per scheduler decoding
// whole rows the conversion took ~4x the sub-stage's MMA time).  Two accumulator buffers (256
// columns each, 128 swapped) let the epilogue overlap the next tile.
//   GEMM1 epilogue: g, u (times their tensor scales) -> the activation -> h rounded to BF16
//                   (row-major [rows, I], expert order: the next GEMM's A operand);
//   GEMM2 epilogue: (acc * ts_down) * router weight, reduced into the token's FP32 output row.
// Every wait is bounded and reports MOE_ERR_DEVICE_TIMEOUT; after a timeout the copies already
// issued are waited for before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kEpiWarps = 4;
constexpr int kCopyWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kConvWarp0 = 6;
constexpr int kConvWarps = 8;   // two per 32-row slice of the tile: half a row each
constexpr int kThreads = (kConvWarp0 + kConvWarps) * 32;
constexpr int kSubK = 64;
constexpr int kTileBytes16 = 128 * 128;       // 128 rows x 64 BF16
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxSegTable = 1027;            // s_tile + s_seg entries the layout reserves

// Shared memory: kSubStages converted sub-stages of K = 64 (the decoded weight tile and the
// token rows: a 256-row tile, two 128-row MMA operands sharing the weight tile; swapped, a 16-row
// tile), a ring of raw NVFP4 weight blocks, barriers, the swapped W4A8 amax exchange and the tile
// tables.  A converted sub-stage waits for its MMAs' completion before the converters may refill
// it, and four did not cover that round trip in the swapped layout, whose sub-stages are as small
// as a raw block: it holds ten.
template <bool kSwap>
struct W16Layout {
  static constexpr int kTokRows = kSwap ? kDecodeTileRows : 2 * kBM;
  static constexpr int kTokBytes = kSubK * kTokRows * 2;
  static constexpr int kSubBytes = kTileBytes16 + kTokBytes;
  static constexpr int kWgtOff = kSwap ? 0 : kTokBytes;   // within a sub-stage
  static constexpr int kTokOff = kSwap ? kTileBytes16 : 0;
  static constexpr int kSubStages = kSwap ? 10 : 3;
  static constexpr int kRawStages = 2;
  // accumulator buffers: 128 rows x (swapped: up to 128 token columns; else two 128-column halves)
  static constexpr uint32_t kAccCols = kSwap ? kBN : 2 * kBN;
  static constexpr uint32_t kTmemCols = 2 * kAccCols;
  static constexpr int kRawOff = kSubStages * kSubBytes;
  static constexpr int kBarOff = kRawOff + kRawStages * kTileBlockBytes;
  static constexpr int kAmaxOff = kBarOff + 512;   // swapped W4A8 GEMM1: [2][kEpiWarps][16] FP32
  static constexpr int kTableOff = kAmaxOff + 2 * kEpiWarps * 16 * 4;
  static constexpr size_t kSmemFixed = 1024 + kTableOff;
  static_assert(kSubBytes % 1024 == 0 && kRawOff % 1024 == 0 && kTileBlockBytes % 1024 == 0,
                "1024-byte aligned tiles");
  static_assert(kSmemFixed + 8 * kMaxSegTable <= 232448, "shared memory");
  // raw full/empty, sub full/empty, acc full/empty x2, drain, 2 epilogue pairs x 2; TMEM slot,
  // issue and arrival counts
  static_assert((2 * kRawStages + 2 * kSubStages + 4 + 1 + 4) * 8 + (4 + kConvWarps) * 4 <= 512,
                "barrier area");
};

// Instruction descriptor of tcgen05.mma kind::f16: FP32 accumulator (bits 4-5 = 1), A and B BF16
// (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Eight E2M1 codes (a 32-bit word, the first code in the low nibble) as four BF16x2 words of
// their values times 2^-126, by placing bits: a code's three magnitude bits (e1 e0 m) become the
// two lowest exponent bits and the top mantissa bit of a BF16, its sign bit the sign.  With
// e1 e0 = 0 that is the subnormal m * 2^-127 = (m / 2) * 2^-126, otherwise
// 2^(e - 127) * (1 + m / 2) = 2^(e - 1) * (1 + m / 2) * 2^-126: E2M1's own definition, scaled.
// Word i holds codes 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void e2m1x8_to_bf16x2_scaled_down(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t ev = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6: the low nibble of each byte
  const uint32_t od = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // byte 0 <- byte i of ev, byte 2 <- byte i of od, bytes 1 and 3 <- the sign of ev's byte 0
    // (selector 8), which is clear: code 2i in bits 0-3 and code 2i+1 in bits 16-19
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;"
        : "=r"(r)
        : "r"(ev), "r"(od), "r"(0x8080u | (uint32_t)i | ((uint32_t)(4 + i) << 8)));
    // magnitude to bits 6-8 (x 2^6) and sign to bit 15 (x 2^12) of each half; the two shifted
    // copies occupy disjoint bits, so the sum is their union
    o[i] = (r * 4160u) & 0x81C081C0u;
  }
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

constexpr uint32_t kBf16x2Pow2_126 = 0x7E807E80u;   // 2^126 in both halves
constexpr uint32_t kBf16x2Pow2_120 = 0x7B807B80u;   // 2^120 in both halves

constexpr uint32_t kBf16x2Pow2_118 = 0x7A807A80u;   // 2^118 in both halves

// An E4M3 block scale times 2^118 as BF16x2 (exact; at most 448 * 2^118 < 2^127): its seven
// magnitude bits shifted to the top of a BF16's exponent-and-mantissa field are the scale times
// 2^-120 (subnormal E4M3 to subnormal BF16 likewise), then two multiplications by powers of two.
// Times an E2M1 value placed at 2^-126 this gives the product times 2^-8, at least 2^-19: a
// normal BF16, exact, and only a power of two away from the decoded weight.
__device__ __forceinline__ uint32_t e4m3_scale_x2118_bf16x2(uint32_t b) {
  const uint32_t h = ((b & 0x7Fu) << 4) | ((b & 0x80u) << 8);
  return mul_bf16x2(mul_bf16x2(h | (h << 16), kBf16x2Pow2_120), kBf16x2Pow2_118);
}

// NVFP4 weights sit in the BF16 tile times 2^-8; the epilogue's tensor scales take the 2^8 back
// (a power of two: the FP32 accumulator is the exact-weight accumulator times 2^-8, bit for bit,
// unless a product falls below 2^-118 into FP32's subnormal range).
template <bool kMx>
__device__ __forceinline__ float weight_tile_comp() {
  return kMx ? 1.0f : 256.0f;
}

// An E8M0 block scale 2^(b - 127) as BF16x2: the byte is the BF16 exponent field (b = 0: the
// subnormal 2^-127).
__device__ __forceinline__ uint32_t e8m0_scale_bf16x2(uint32_t b) {
  const uint32_t h = b ? (b << 7) : 0x40u;
  return h | (h << 16);
}

struct TileW16 {
  int seg, m0, rows, nt;
};

__device__ __forceinline__ TileW16 decode_tile_w16(int item, int n_tiles, const int32_t* s_tile,
                                                   const int32_t* s_seg, int nseg, int tr) {
  TileW16 t;
  const int mt = item / n_tiles;
  t.nt = item - mt * n_tiles;
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tile[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  t.seg = lo;
  t.m0 = s_seg[lo] + (mt - s_tile[lo]) * tr;
  t.rows = min(tr, s_seg[lo + 1] - t.m0);
  return t;
}

// MXFP8 requantisation of 32 consecutive h values: E8M0 scale, E4M3 codes (nearest even,
// saturated), and the decoded values as BF16 (exact) for the next GEMM.
__device__ __forceinline__ void mx8_requant_store(const float* h, uint8_t* codes, uint8_t* sf,
                                                  uint8_t* hb) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
  const uint32_t sb = mx_scale_byte(amax, 8);
  const float X = e8m0_to_f32(sb);
  uint32_t cw[8], bw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c2 = f32_to_e4m3x2(mx_unscale(h[2 * i], sb), mx_unscale(h[2 * i + 1], sb));
    if (i & 1) cw[i >> 1] |= c2 << 16;
    else cw[i >> 1] = c2;
    const float2 v = e4m3x2_to_f32x2(c2);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x * X, v.y * X);
    bw[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint4* cd = reinterpret_cast<uint4*>(codes);
  cd[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  cd[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  *sf = (uint8_t)sb;
  uint4* bd = reinterpret_cast<uint4*>(hb);
#pragma unroll
  for (int q = 0; q < 4; ++q) bd[q] = make_uint4(bw[4 * q], bw[4 * q + 1], bw[4 * q + 2], bw[4 * q + 3]);
}

// kSwap (decode-sized batches): the decoded weight tile is the MMA's A operand (M = 128) and a
// tile of kDecodeTileRows expert-ordered token rows its B operand (N = 16), so neither the MMA
// nor the token copies carry the padding of a 128-row token tile; the accumulator holds
// D[weight row][token] and the epilogue works per token column.
template <bool kMx, bool kSwap>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_w16_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmW16Args p) {
  using L = W16Layout<kSwap>;
  constexpr int kTR = L::kTokRows;                               // token rows per tile
  constexpr uint32_t kBoxBytes = (uint32_t)kSubK * kTR * 2;      // one sub-stage's token box
  constexpr uint32_t kTokOff = L::kTokOff, kWgtOff = L::kWgtOff;
  constexpr int kRawStages = L::kRawStages, kSubBytes = L::kSubBytes, kRawOff = L::kRawOff;
  constexpr int kSubStages = L::kSubStages;
  constexpr uint32_t kAccCols = L::kAccCols, kTmemCols = L::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  // the 1024-byte-aligned base, reached by pointer arithmetic on the shared array so that the
  // compiler keeps the shared address space (shared loads and stores, not generic ones)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRawStages;
  uint64_t* sub_full = raw_empty + kRawStages;
  uint64_t* sub_empty = sub_full + kSubStages;
  uint64_t* acc_full = sub_empty + kSubStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* pair_bar = drain + 1;   // [warp pair][tile parity]: swapped W4A8 amax exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 4);
  uint32_t* s_issued = tmem_slot + 1;   // [0] raw blocks, [1] A boxes issued by the copy thread
  uint32_t* s_conv = s_issued + 2;      // sub-stage arrivals of each converter warp
  volatile uint32_t* s_abort = s_conv + kConvWarps;   // set by any role whose wait ran out
  float* s_amax = reinterpret_cast<float*>(smem + L::kAmaxOff);
  int32_t* s_tile = reinterpret_cast<int32_t*>(smem + L::kTableOff);
  int32_t* s_seg = s_tile + (p.nseg + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(smem_u32(raw_full + s), 1);            // the bulk copy (expect_tx)
      mbar_init(smem_u32(raw_empty + s), kConvWarps);  // every converter warp is done with it
    }
    for (int s = 0; s < kSubStages; ++s) {
      mbar_init(smem_u32(sub_full + s), 1 + kConvWarps);   // the A box (expect_tx) + converters
      mbar_init(smem_u32(sub_empty + s), 1);               // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(pair_bar + i), 2);
    s_issued[0] = s_issued[1] = 0u;
    for (int w = 0; w < kConvWarps; ++w) s_conv[w] = 0u;
    *s_abort = 0u;
    fence_barrier_init();
  }
  if (warp == kCopyWarp && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_a) : "memory");
  griddep_wait();
  griddep_launch();
  for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) s_seg[i] = p.seg_off[i];
  {
    // tiles of kTR rows per segment: a prefix over ceil(rows / kTR), one warp (lane l takes a
    // run of consecutive segments)
    __syncthreads();
    if (warp == 0) {
      const int per = (p.nseg + 31) / 32;
      const int s0 = min(lane * per, p.nseg), s1 = min(s0 + per, p.nseg);
      int c = 0;
      for (int i = s0; i < s1; ++i) c += (max(s_seg[i + 1] - s_seg[i], 0) + kTR - 1) / kTR;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int off = incl - c;
      for (int i = s0; i < s1; ++i) {
        s_tile[i] = off;
        off += (max(s_seg[i + 1] - s_seg[i], 0) + kTR - 1) / kTR;
      }
      if (lane == 31) s_tile[p.nseg] = incl;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_tiles = p.N / kBN;
  int total = s_tile[p.nseg] * n_tiles;
  if (total < 0 || total > p.max_items) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_INVALID_ARG);
    total = 0;
  }
  const int kblk = p.K / kBK;        // raw weight blocks per tile
  const uint32_t smem0 = smem_u32(smem);

  if (warp == kCopyWarp) {
    // ---------------- raw weight blocks (bulk) and activation boxes (TMA) ----------------
    if (lane == 0) {
      int rs = 0, ss = 0;
      uint32_t rph = 0, sph = 0, n_raw = 0, n_sub = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const TileW16 t = decode_tile_w16(item, n_tiles, s_tile, s_seg, p.nseg, kTR);
        const uint8_t* bsrc = p.b_tiles + (size_t)t.seg * p.b_per_seg +
                              (size_t)t.nt * kblk * kTileBlockBytes;
        for (int kb = 0; kb < kblk && ok; ++kb) {
          if (!mbar_wait_bounded(smem_u32(raw_empty + rs), rph ^ 1u, kWaitLimitNs, p.status)) {
            ok = false;
            break;
          }
          const uint32_t rb = smem_u32(raw_full + rs);
          mbar_arrive_expect_tx(rb, kTileBlockBytes);
          bulk_load(smem0 + kRawOff + rs * kTileBlockBytes, bsrc + (size_t)kb * kTileBlockBytes,
                    kTileBlockBytes, rb);
          ++n_raw;
          if (++rs == kRawStages) { rs = 0; rph ^= 1u; }
          for (int q = 0; q < kBK / kSubK; ++q) {
            if (!mbar_wait_bounded(smem_u32(sub_empty + ss), sph ^ 1u, kWaitLimitNs, p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(sub_full + ss);
            mbar_arrive_expect_tx(fb, kBoxBytes);
            tma_load_2d(smem0 + ss * kSubBytes + kTokOff, &tmap_a, kb * kBK + q * kSubK, t.m0, fb);
            ++n_sub;
            if (++ss == kSubStages) { ss = 0; sph ^= 1u; }
          }
        }
      }
      s_issued[0] = n_raw;
      s_issued[1] = n_sub;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp >= kConvWarp0) {
    // ---------------- NVFP4 weight row -> BF16 row of the B tile ----------------
    const int cwarp = warp - kConvWarp0;
    const int r = (cwarp & 3) * 32 + lane;   // weight row of the tile
    const int hf = cwarp >> 2;               // which half of the sub-stage's 64 codes
    int rs = 0, ss = 0;
    uint32_t rph = 0, sph = 0, n_arr = 0;
    bool ok = true;
    // byte offsets of this thread's 16-byte code chunk 2q + hf of row r (stored at chunk ^ (r % 8))
    uint32_t coff[kBK / kSubK];
#pragma unroll
    for (int q = 0; q < kBK / kSubK; ++q) coff[q] = r * 128 + (((2 * q + hf) ^ (r & 7)) << 4);
    // NVFP4: the four E4M3 scales of the row's sub-stage q are one word of scale group q
    const uint32_t soff = kTileBytes + (r & 31) * 16 + (r >> 5) * 4;
    uint8_t* const wtile = smem + kWgtOff + r * 128;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      for (int kb = 0; kb < kblk && ok; ++kb) {
        // every lane waits; the decision is made together, so the warp never diverges
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(raw_full + rs), rph,
                                                       kWaitLimitNs, p.status))) {
          ok = false;
          break;
        }
        // the thread's codes and scales of the whole block go to registers, and the block's
        // slot is handed back before any of it is decoded
        const uint8_t* raw = smem + kRawOff + rs * kTileBlockBytes;
        uint4 cq[kBK / kSubK];
        uint32_t sq[kBK / kSubK];
#pragma unroll
        for (int q = 0; q < kBK / kSubK; ++q) {
          cq[q] = *reinterpret_cast<const uint4*>(raw + coff[q]);
          // MXFP4: E8M0 scale 2q + hf of the row's eight covers this chunk's 32 codes
          sq[q] = kMx ? raw[kTileBytes + r * 8 + 2 * q + hf]
                      : *reinterpret_cast<const uint32_t*>(raw + soff + q * 512);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(raw_empty + rs));
        if (++rs == kRawStages) { rs = 0; rph ^= 1u; }
#pragma unroll
        for (int q = 0; q < kBK / kSubK; ++q) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(sub_empty + ss), sph ^ 1u,
                                                         kWaitLimitNs, p.status))) {
            ok = false;
            break;
          }
          // the multipliers of the chunk's values (times 2^-126 after the bit placement):
          // NVFP4: 16-blocks 2hf (16-byte output chunks 4hf, 4hf+1) and 2hf+1 (4hf+2, 4hf+3), each
          // times 2^118, so the tile holds the weights times 2^-8 (restored in the epilogue);
          // MXFP4: 2^126 and the one E8M0 scale of the chunk, applied one after the other
          uint32_t m0, m1;
          if constexpr (kMx) {
            m0 = e8m0_scale_bf16x2(sq[q]);
            m1 = m0;
          } else {
            m0 = e4m3_scale_x2118_bf16x2((sq[q] >> (16 * hf)) & 0xFFu);
            m1 = e4m3_scale_x2118_bf16x2((sq[q] >> (16 * hf + 8)) & 0xFFu);
          }
          const uint32_t cw[4] = {cq[q].x, cq[q].y, cq[q].z, cq[q].w};
          uint8_t* brow = wtile + ss * kSubBytes;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {      // 16-byte chunk j of the BF16 row: 8 values
            const int j = 4 * hf + jj;
            const uint32_t m = jj < 2 ? m0 : m1;
            uint32_t v[4];
            e2m1x8_to_bf16x2_scaled_down(cw[jj], v);
            uint4 o;
            if constexpr (kMx) {
              o.x = mul_bf16x2(mul_bf16x2(v[0], kBf16x2Pow2_126), m);
              o.y = mul_bf16x2(mul_bf16x2(v[1], kBf16x2Pow2_126), m);
              o.z = mul_bf16x2(mul_bf16x2(v[2], kBf16x2Pow2_126), m);
              o.w = mul_bf16x2(mul_bf16x2(v[3], kBf16x2Pow2_126), m);
            } else {
              o.x = mul_bf16x2(v[0], m);
              o.y = mul_bf16x2(v[1], m);
              o.z = mul_bf16x2(v[2], m);
              o.w = mul_bf16x2(v[3], m);
            }
            *reinterpret_cast<uint4*>(brow + ((j ^ (r & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();     // the tensor core reads what these stores wrote
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(sub_full + ss));
          ++n_arr;
          if (++ss == kSubStages) { ss = 0; sph ^= 1u; }
        }
      }
    }
    if (lane == 0) {
      s_conv[warp - kConvWarp0] = n_arr;
      if (!ok) *s_abort = 1u;
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = kSwap ? make_idesc_bf16(128, kTR) : make_idesc_bf16(kBM, kBN);
      int ss = 0;
      uint32_t sph = 0;
      uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
      // A: the token rows (or, kSwap, the decoded weights); B: the other tile of the sub-stage
      const uint64_t dA0 = smem_desc(smem0 + (kSwap ? kWgtOff : kTokOff), 16, 1024,
                                     kLayoutSwizzle128B);
      const uint64_t dB0 = smem_desc(smem0 + (kSwap ? kTokOff : kWgtOff), 16, 1024,
                                     kLayoutSwizzle128B);
      bool ok = true;
      int it = 0;
      const int nsub = kblk * (kBK / kSubK);
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
        for (int k = 0; k < nsub; ++k) {
          if (!mbar_wait_bounded(smem_u32(sub_full + ss), sph, kWaitLimitNs, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((uint32_t)(ss * kSubBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kSubK / 16; ++kk) {   // K = 16 per MMA: 32 bytes -> 2 units
            tc_mma_bf16(d_tmem, dA0 + so + kk * 2, dB0 + so + kk * 2, idesc,
                        (k | kk) != 0 ? 1u : 0u);
            if constexpr (!kSwap)   // token rows 128-255 (16 KB further) into the second half
              tc_mma_bf16(d_tmem + kBN, dA0 + so + (kTileBytes16 >> 4) + kk * 2, dB0 + so + kk * 2,
                          idesc, (k | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(sub_empty + ss));
          if (++ss == kSubStages) { ss = 0; sph ^= 1u; }
        }
        if (ok) tc_commit(smem_u32(acc_full + abuf));
      }
      tc_commit(smem_u32(drain));
      if (!mbar_wait_bounded(smem_u32(drain), 0u, kWaitLimitNs, p.status)) ok = false;
      if (!ok) *s_abort = 1u;
    }
  } else if constexpr (kSwap) {
    // ---------------- epilogue (warps 0-3), swapped: lane = weight row, column = token ----------
    uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
    int it = 0;
    const int r = warp * 32 + lane;
    const bool lo = lane < 16;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      const TileW16 t = decode_tile_w16(item, n_tiles, s_tile, s_seg, p.nseg, kTR);
      const int abuf = it & 1;
      const uint32_t acc_par = (acc_phase >> abuf) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_full + abuf), acc_par,
                                                     kWaitLimitNs, p.status))) {
        if (lane == 0) *s_abort = 1u;
        break;
      }
      acc_phase ^= 1u << abuf;
      tc_fence_after();
      uint32_t v[16];
      tmem_ld_32x32b_x16(tmem_base + abuf * kAccCols + ((uint32_t)(warp * 32) << 16), v);
      tmem_ld_wait();
      // the accumulator is in registers: the buffer goes back before the stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + abuf));
      // valid token columns 0 .. nrow-1 (none if malformed segment offsets put the tile outside
      // the expert-ordered rows)
      const int nrow = t.m0 < 0 ? 0 : min(t.rows, p.out_rows - t.m0);
      if (p.mode == 0) {
        const bool gated = p.act != kActRelu2;
        const int I = gated ? p.N / 2 : p.N;
        const float ag = p.w_ts[t.seg * 4 + 0] * weight_tile_comp<kMx>();
        const float au = p.w_ts[t.seg * 4 + 1] * weight_tile_comp<kMx>();
        __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(p.hb);
        if (gated) {
          // rows 32w .. 32w+15 are the gates and 32w+16 .. 32w+31 the ups of features
          // 16w .. 16w+15 of the tile's 64: lane l takes tokens 8 (l / 16) .. +7 of feature
          // l % 16 with its partner lane's half of the pair
          const int j0 = lo ? 0 : 8;
          const int f = t.nt * (kBN / 2) + warp * 16 + (lane & 15);
          float h[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t got = __shfl_xor_sync(0xffffffffu, lo ? v[8 + j] : v[j], 16);
            const float g = __uint_as_float(lo ? v[j] : got);
            const float u = __uint_as_float(lo ? got : v[8 + j]);
            h[j] = glu_activation(g * ag, u * au, p.act, p.swiglu_limit, p.swiglu_alpha);
          }
          if constexpr (kMx) {
            // a 32-feature MXFP8 block spans warps 2i and 2i+1: the amax of each token over
            // the warp's 16 features, then over the pair through shared memory
            float am[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              am[j] = fabsf(h[j]);
#pragma unroll
              for (int o = 1; o < 16; o <<= 1)
                am[j] = fmaxf(am[j], __shfl_xor_sync(0xffffffffu, am[j], o));
            }
            float* mine = s_amax + (abuf * kEpiWarps + warp) * 16;
            if ((lane & 15) == 0)
#pragma unroll
              for (int j = 0; j < 8; ++j) mine[j0 + j] = am[j];
            __syncwarp();
            const uint32_t pb = smem_u32(pair_bar + (warp >> 1) * 2 + abuf);
            if (lane == 0) mbar_arrive(pb);
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(pb, (uint32_t)(it >> 1) & 1u,
                                                           kWaitLimitNs, p.status))) {
              if (lane == 0) *s_abort = 1u;
              break;
            }
            const float* other = s_amax + (abuf * kEpiWarps + (warp ^ 1)) * 16;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (j0 + j >= nrow) continue;
              const size_t prow = (size_t)(t.m0 + j0 + j);
              const uint32_t sb = mx_scale_byte(fmaxf(am[j], other[j0 + j]), 8);
              const uint32_t code = f32_to_e4m3x2(mx_unscale(h[j], sb), 0.0f) & 0xFFu;
              p.hq8[prow * I + f] = (uint8_t)code;
              hb[prow * I + f] = __float2bfloat16_rn(e4m3x2_to_f32x2(code).x * e8m0_to_f32(sb));
              if ((lane & 15) == 0 && (warp & 1) == 0) p.hsf8[prow * (I / 32) + f / 32] = (uint8_t)sb;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (j0 + j < nrow)
                hb[(size_t)(t.m0 + j0 + j) * I + f] = __float2bfloat16_rn(h[j]);
          }
        } else {
          // non-gated: row r is feature r of the tile's 128, 16 tokens per lane; a warp's 32
          // features are one MXFP8 block
          const int f = t.nt * kBN + r;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float hv = glu_activation(0.0f, __uint_as_float(v[j]) * au, p.act,
                                            p.swiglu_limit, p.swiglu_alpha);
            const size_t prow = (size_t)(t.m0 + j);
            if constexpr (kMx) {
              float am = fabsf(hv);
#pragma unroll
              for (int o = 1; o < 32; o <<= 1)
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
              if (j >= nrow) continue;
              const uint32_t sb = mx_scale_byte(am, 8);
              const uint32_t code = f32_to_e4m3x2(mx_unscale(hv, sb), 0.0f) & 0xFFu;
              p.hq8[prow * I + f] = (uint8_t)code;
              hb[prow * I + f] = __float2bfloat16_rn(e4m3x2_to_f32x2(code).x * e8m0_to_f32(sb));
              if (lane == 0) p.hsf8[prow * (I / 32) + f / 32] = (uint8_t)sb;
            } else {
              if (j < nrow) hb[prow * I + f] = __float2bfloat16_rn(hv);
            }
          }
        }
      } else {
        // lane j < 16 fetches the token and router weight of the tile's row j
        const float alpha = p.w_ts[t.seg * 4 + 2] * weight_tile_comp<kMx>();
        int tok = -1;
        float wr = 0.0f;
        if (lane < nrow) {
          tok = __ldg(p.perm_src + t.m0 + lane);
          wr = __ldg(p.perm_w + t.m0 + lane);
          if (tok < 0 || tok >= p.y_rows) {
            set_status(p.status, MOE_ERR_INVALID_ARG);
            tok = -1;
          }
        }
        float* ycol = p.yacc + t.nt * kBN + r;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tj = __shfl_sync(0xffffffffu, tok, j);
          const float wj = __shfl_sync(0xffffffffu, wr, j);
          if (tj >= 0) atomicAdd(ycol + (size_t)tj * p.N, (__uint_as_float(v[j]) * alpha) * wj);
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 0-3): one accumulator row per thread ----------------
    uint32_t acc_phase = 0u;   // bit b: the phase of accumulator buffer b
    int it = 0;
    const int r = warp * 32 + lane;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      const TileW16 t = decode_tile_w16(item, n_tiles, s_tile, s_seg, p.nseg, kTR);
      const int abuf = it & 1;
      const uint32_t acc_par = (acc_phase >> abuf) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_full + abuf), acc_par,
                                                     kWaitLimitNs, p.status))) {
        if (lane == 0) *s_abort = 1u;
        break;
      }
      acc_phase ^= 1u << abuf;
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {   // token rows 0-127, then 128-255 of the tile
        const int prow = t.m0 + half * kBM + r;
        const bool valid = half * kBM + r < t.rows && prow >= 0 && prow < p.out_rows;
        const uint32_t tbase =
            tmem_base + abuf * kAccCols + half * kBN + ((uint32_t)(warp * 32) << 16);
        if (p.mode == 0) {
          const bool gated = p.act != kActRelu2;
          const int I = gated ? p.N / 2 : p.N;
          const float ag = p.w_ts[t.seg * 4 + 0] * weight_tile_comp<kMx>();
          const float au = p.w_ts[t.seg * 4 + 1] * weight_tile_comp<kMx>();
          float hk[16];   // W4A8, gated: the first 16 features of a 32-feature MXFP8 block
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
            if (!valid) continue;
            if constexpr (kMx) {
              float h32[32];
              if (gated) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float hv = glu_activation(__uint_as_float(v[i]) * ag,
                                                  __uint_as_float(v[16 + i]) * au, p.act,
                                                  p.swiglu_limit, p.swiglu_alpha);
                  if (c & 1) h32[16 + i] = hv;
                  else hk[i] = hv;
                }
                if ((c & 1) == 0) continue;
#pragma unroll
                for (int i = 0; i < 16; ++i) h32[i] = hk[i];
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  h32[i] = glu_activation(0.0f, __uint_as_float(v[i]) * au, p.act, p.swiglu_limit,
                                          p.swiglu_alpha);
              }
              const int f0 = gated ? t.nt * (kBN / 2) + (c - 1) * 16 : t.nt * kBN + c * 32;
              mx8_requant_store(h32, p.hq8 + (size_t)prow * I + f0,
                                p.hsf8 + (size_t)prow * (I / 32) + f0 / 32,
                                p.hb + ((size_t)prow * I + f0) * 2);
              continue;
            }
            // gated: (16 gate | 16 up) columns -> 16 features; non-gated: 32 up columns -> 32
            uint32_t packed[16];
            if (gated) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float h0 = glu_activation(__uint_as_float(v[2 * i]) * ag,
                                                __uint_as_float(v[16 + 2 * i]) * au, p.act,
                                                p.swiglu_limit, p.swiglu_alpha);
                const float h1 = glu_activation(__uint_as_float(v[2 * i + 1]) * ag,
                                                __uint_as_float(v[17 + 2 * i]) * au, p.act,
                                                p.swiglu_limit, p.swiglu_alpha);
                const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
                packed[i] = *reinterpret_cast<const uint32_t*>(&b);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float h0 = glu_activation(0.0f, __uint_as_float(v[2 * i]) * au, p.act,
                                                p.swiglu_limit, p.swiglu_alpha);
                const float h1 = glu_activation(0.0f, __uint_as_float(v[2 * i + 1]) * au, p.act,
                                                p.swiglu_limit, p.swiglu_alpha);
                const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
                packed[i] = *reinterpret_cast<const uint32_t*>(&b);
              }
            }
            const int f0 = gated ? t.nt * (kBN / 2) + c * 16 : t.nt * kBN + c * 32;
            uint4* dst = reinterpret_cast<uint4*>(p.hb + ((size_t)prow * I + f0) * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (i < (gated ? 2 : 4))
                dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                    packed[4 * i + 3]);
          }
        } else {
          const float alpha = p.w_ts[t.seg * 4 + 2] * weight_tile_comp<kMx>();
          int tok = 0;
          float wr = 0.0f;
          bool ok_row = valid;
          if (valid) {
            tok = __ldg(p.perm_src + prow);
            wr = __ldg(p.perm_w + prow);
            if (tok < 0 || tok >= p.y_rows) {
              set_status(p.status, MOE_ERR_INVALID_ARG);
              ok_row = false;
            }
          }
          float* yrow = p.yacc + (size_t)(ok_row ? tok : 0) * p.N + t.nt * kBN;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + c * 32, v);
            tmem_ld_wait();
            if (!ok_row) continue;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              red_add_v4(yrow + c * 32 + 4 * i, (__uint_as_float(v[4 * i]) * alpha) * wr,
                         (__uint_as_float(v[4 * i + 1]) * alpha) * wr,
                         (__uint_as_float(v[4 * i + 2]) * alpha) * wr,
                         (__uint_as_float(v[4 * i + 3]) * alpha) * wr);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + abuf));
    }
  }

  // Teardown.  After a timeout, copies into shared memory may still be in flight.  A sub-stage
  // completes on the A box (copy thread, with its bytes) and one arrival per converter warp;
  // every participant waits for the slot's release before it arrives, so only the last
  // kSubStages indices can be open, and the arrivals missing there are made here on behalf of
  // whoever stopped, after which every issued phase completes once its bytes land.  Then the
  // last phases of both rings are waited for (bounded).  Without a timeout every phase was
  // consumed, and none of this runs.
  tc_fence_before();
  __syncthreads();
  if (*s_abort && warp == kCopyWarp && lane == 0) {
    const uint32_t nr = s_issued[0], na = s_issued[1];
    uint32_t hi = na;
    for (int w = 0; w < kConvWarps; ++w) hi = max(hi, s_conv[w]);
    const uint32_t lo = hi > (uint32_t)kSubStages ? hi - kSubStages : 0u;
    for (uint32_t i = lo; i < hi; ++i) {
      const uint32_t bar = smem_u32(sub_full + i % kSubStages);
      if (i >= na) mbar_arrive(bar);
      for (int w = 0; w < kConvWarps; ++w)
        if (i >= s_conv[w]) mbar_arrive(bar);
    }
    for (uint32_t i = lo; i < hi; ++i)
      if (!mbar_wait_bounded(smem_u32(sub_full + i % kSubStages), (i / kSubStages) & 1u,
                             kWaitLimitNs, p.status))
        break;
    for (uint32_t i = nr > (uint32_t)kRawStages ? nr - kRawStages : 0u; i < nr; ++i)
      if (!mbar_wait_bounded(smem_u32(raw_full + i % kRawStages), (i / kRawStages) & 1u,
                             kWaitLimitNs, p.status))
        break;
  }
  if (*s_abort) {
    tc_fence_before();
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_w16() {
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

cudaError_t launch_grouped_gemm_w16(const GemmW16Args& a, cudaStream_t s) {
  auto encode = encode_fn_w16();
  if (!encode) return cudaErrorNotSupported;
  if (a.N % kBN != 0 || a.K % kBK != 0 || a.nseg < 1) return cudaErrorInvalidValue;
  // expert-ordered BF16 rows [out_rows, K]; box = 64 elements (128 bytes) x the tile's token rows
  // (256, or kDecodeTileRows swapped)
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.out_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kSubK, (cuuint32_t)(a.swap ? W16Layout<true>::kTokRows
                                                                    : W16Layout<false>::kTokRows)};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.a_rows), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (a.nseg + 2 > kMaxSegTable) return cudaErrorInvalidValue;
  const size_t smem = (a.swap ? W16Layout<true>::kSmemFixed : W16Layout<false>::kSmemFixed) +
                      sizeof(int32_t) * 2 * ((size_t)a.nseg + 2);
  auto kernel = a.mx ? (a.swap ? grouped_gemm_w16_kernel<true, true>
                               : grouped_gemm_w16_kernel<true, false>)
                     : (a.swap ? grouped_gemm_w16_kernel<false, true>
                               : grouped_gemm_w16_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int grid = a.max_items;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, tmap, a);
}

}  // namespace nvfp4moe
