// Internal declarations of the NVFP4 MoE library: buffer layouts and kernel launchers.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "nvfp4_moe.h"

namespace nvfp4moe {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// GEMM tiling shared by the host and the kernels.
constexpr int kBM = 128;       // permuted rows per tile (MMA M)
constexpr int kBN = 128;       // output columns per tile (MMA N)
constexpr int kBK = 256;       // FP4 elements of K per pipeline stage (128 bytes per row)
constexpr int kMmaK = 64;      // K of one block-scaled FP4 MMA
constexpr int kDecodeMaxRows = 64;   // batches up to this many tokens take the decode path
constexpr int kDecodeTileRows = 16;  // rows of an expert per decode GEMM tile (its MMA N)
constexpr int kSmallPlanRows = 2048; // T*k routed by the one-block plan

// Activation of GEMM1's epilogue (GemmArgs::act).
constexpr int kActSwiglu = 0;        // silu(g) * u
constexpr int kActSwigluClamp = 1;   // silu(min(g, L)) * clamp(u, -L, L)
constexpr int kActRelu2 = 2;         // max(u, 0)^2, non-gated experts
constexpr int kActSwigluOai = 3;     // (clamp(u, -L, L) + 1) * g' * sigmoid(alpha * g'), g' = min(g, L)

// Router chunking: tokens per chunk (one router block and one scatter block each).
inline int plan_tokens_per_chunk(int k) { return k <= 16 ? 64 : 32; }

// Private layout of the packed-weight buffer: every weight matrix is stored as GEMM-ready
// blocks, one per (128-row N tile, 256-wide K stage), each block 18432 contiguous bytes:
//   [0, 16384)      codes of the 128 rows x 128 bytes, row r at r*128, its 16-byte chunk c stored
//                   at chunk position c ^ (r % 8) (the 128-byte swizzle the MMA descriptor uses);
//   [16384, 18432)  E4M3 scales as four 512-byte groups (one per 64-wide MMA K step), row r's
//                   scale word (4 scales) at (r % 32)*16 + (r / 32)*4 (the arrangement that the
//                   tensor-memory scale copy expects).
// A tile of the MMA's B operand for one pipeline stage is therefore one contiguous bulk copy.
//   w13 [Et][2I/128][H/256][18432]: GEMM1 rows interleaved by 16 (rows 32b+i are gate rows
//       16b+i for i < 16, up rows 16b+i-16 otherwise); for non-gated experts (ReLU2)
//       [Et][I/128][H/256][18432], the up rows in order;
//   w2  [Et][H/128][I/256][18432]: GEMM2 (down) rows;
//   ts  [Et][4] FP32: gate, up, down tensor scales (the 4th is padding);
//   bias [E] FP32: the variant router's per-expert selection bias (zero unless set).
// Et = E + 1 with a shared expert, which is stored last.
constexpr int kTileBytes = 128 * 128;             // codes of one (N tile, K stage) block
constexpr int kTileSfBytes = 4 * 512;             // its scales
constexpr int kTileBlockBytes = kTileBytes + kTileSfBytes;

// Widths that are multiples of 32 but not of the K stage (256) run at the next multiple of 256:
// weights are packed with zero rows and columns up to it, and x (or its codes) is copied into a
// zero-padded row of the workspace.  A padded column of x meets only zero weights, a padded
// weight row yields h = activation(0, 0) = 0 for every activation of the layer (quantised to a
// zero block), and a padded output column is never copied out, so every sum of the layer takes
// exactly the same nonzero terms as the unpadded definition.
// A shared expert whose intermediate size differs from the routed experts' runs at the same
// padded width: both are padded to the next multiple of 256 above the larger of the two.
inline int pad_stage(int v) { return (v + 255) / 256 * 256; }
inline int h_width(const moe_config& c) {   // the widest intermediate of the layer
  return c.shared_inter > c.inter ? c.shared_inter : c.inter;
}
inline bool needs_padding(const moe_config& c) {
  return c.hidden % 256 != 0 || c.inter % 256 != 0 ||
         (c.shared_inter > 0 && c.shared_inter != c.inter);
}
inline moe_config padded_config(const moe_config& c) {
  moe_config p = c;
  p.hidden = pad_stage(c.hidden);
  p.inter = pad_stage(h_width(c));
  if (c.shared_inter > 0) p.shared_inter = p.inter;
  return p;
}

// GEMM1 output rows per expert: gate and up rows (2I), or the up rows alone for non-gated
// experts (I).
inline bool gated_experts(const moe_config& c) { return (c.flags & MOE_FLAG_ACT_RELU2) == 0u; }
inline int gemm1_rows(const moe_config& c) { return gated_experts(c) ? 2 * c.inter : c.inter; }

struct WeightLayout {
  int E, Et, H, I;
  bool gated;
  size_t w13, w2, ts, bias, total;
  size_t w13_per_e, w2_per_e;
  explicit WeightLayout(const moe_config& c) {
    E = c.num_experts;
    Et = E + (c.shared_inter > 0 ? 1 : 0);
    H = c.hidden;
    I = c.inter;
    gated = gated_experts(c);
    w13_per_e = (size_t)(gemm1_rows(c) / 128) * (H / 256) * kTileBlockBytes;
    w2_per_e = (size_t)(H / 128) * (I / 256) * kTileBlockBytes;
    size_t o = 0;
    w13 = o; o = align_up(o + w13_per_e * Et);
    w2 = o;  o = align_up(o + w2_per_e * Et);
    ts = o;  o = align_up(o + sizeof(float) * 4 * Et);
    bias = o; o = align_up(o + sizeof(float) * E);   // router selection bias (variant router)
    total = o;
  }
};

// Byte offsets of the code byte pair (row n, 16-block kb) and of its scale inside one packed
// matrix with K columns (K a multiple of 256, rows a multiple of 128).
__host__ __device__ __forceinline__ size_t packed_code_offset(int64_t n, int64_t kb, int64_t K) {
  const int64_t kst = K / 256, r = n & 127;
  const int64_t blk = (n >> 7) * kst + kb / 16;
  const int64_t c = (kb % 16) >> 1;               // 16-byte chunk of the 128-byte row slice
  return (size_t)(blk * kTileBlockBytes + r * 128 + ((c ^ (r & 7)) << 4) + (kb & 1) * 8);
}
__host__ __device__ __forceinline__ size_t packed_sf_offset(int64_t n, int64_t kb, int64_t K) {
  const int64_t kst = K / 256, r = n & 127;
  const int64_t blk = (n >> 7) * kst + kb / 16;
  return (size_t)(blk * kTileBlockBytes + kTileBytes + ((kb % 16) >> 2) * 512 + (r & 31) * 16 +
                  (r >> 5) * 4 + (kb & 3));
}

// Small batches run a fused prologue (one block does the quantiser, router and plan) and combine
// by storing every assignment's output row and summing a token's rows in slot order.
constexpr int64_t kSmallPrologueElems = 512 * 1024;   // T*H handled by the one-block prologue
constexpr int64_t kStoreCombineElems = 16 << 20;      // (T*k + shared T) * H stored in FP32
bool prologue_small_fits(int T, int H, int k);

// Workspace of moe_run for T tokens.  Offset 0 holds the device status word.
struct RunLayout {
  size_t hdr, amax_part, ids, w, hist, base, seg_off, tile_start, perm_src, perm_w, inv, xq, xsf,
      hq, hsf, yacc, obuf, perm_seg, xq_perm, xsf_tiles, hsf_tiles, ready, xb_perm, hb, xq8,
      hq8, total;
  int T, R, Rt, nseg, nchunks, tpc, dtiles;
  bool small;   // fused prologue + stored-row combine
  bool decode;  // T <= kDecodeMaxRows: cluster prologue and the swapped-operand decode GEMM
  bool w16;     // W4A16 or W4A8 layer: BF16 activation and h rows (decoded), one path
  bool mx;      // W4A8 layer: MXFP8 codes and scales of x and h as well
  RunLayout(const moe_config& c, int T_) {
    T = T_;
    const int k = c.top_k, E = c.num_experts, H = c.hidden, I = c.inter;
    const int shared = c.shared_inter > 0 ? 1 : 0;
    R = T * k;
    Rt = R + shared * T;
    nseg = E + shared;
    tpc = plan_tokens_per_chunk(k);
    nchunks = (T + tpc - 1) / tpc;
    size_t o = 0;
    hdr = o;        o = align_up(o + 256);
    amax_part = o;  o = align_up(o + 4 * 1024);
    ids = o;        o = align_up(o + 4 * (size_t)R);
    w = o;          o = align_up(o + 4 * (size_t)R);
    hist = o;       o = align_up(o + 4 * ((size_t)nchunks * E + 1 + E));
    base = o;       o = align_up(o + 4 * (size_t)nchunks * E);
    seg_off = o;    o = align_up(o + 4 * (size_t)(nseg + 2));
    tile_start = o; o = align_up(o + 4 * (size_t)(nseg + 2));
    perm_src = o;   o = align_up(o + 4 * (size_t)Rt);
    perm_w = o;     o = align_up(o + 4 * (size_t)Rt);
    inv = o;        o = align_up(o + 4 * (size_t)R);
    xq = o;         o = align_up(o + (size_t)T * H / 2);
    xsf = o;        o = align_up(o + (size_t)T * H / 16);
    hq = o;         o = align_up(o + (size_t)Rt * I / 2);
    hsf = o;        o = align_up(o + (size_t)Rt * I / 16);
    mx = (c.flags & MOE_FLAG_ACT_MXFP8) != 0u;
    w16 = mx || (c.flags & MOE_FLAG_ACT_BF16) != 0u;
    small = !w16 && (int64_t)R <= 2048 && (int64_t)T * H <= kSmallPrologueElems &&
            (int64_t)Rt * H <= kStoreCombineElems;
    yacc = o;       o = align_up(o + (small ? 0 : 4 * (size_t)T * H));
    obuf = o;       o = align_up(o + (small ? 4 * (size_t)Rt * H : 0));
    decode = small && T <= kDecodeMaxRows;
    // m-tiles of expert-ordered rows: 128 rows (general), kDecodeTileRows rows (decode, where an
    // active expert owns ceil(rows / kDecodeTileRows) of them)
    if (decode) {
      const int64_t bound = (int64_t)nseg + (Rt + kDecodeTileRows - 1) / kDecodeTileRows;
      dtiles = (int)(bound < Rt ? bound : Rt);
    } else {
      dtiles = (int)(((int64_t)Rt + (int64_t)nseg * 127) / 128);
    }
    perm_seg = o;   o = align_up(o + 4 * (size_t)Rt);
    xq_perm = o;    o = align_up(o + (size_t)Rt * H / 2);
    xsf_tiles = o;  o = align_up(o + (size_t)dtiles * (H / 64) * 512);
    hsf_tiles = o;  o = align_up(o + (size_t)dtiles * (I / 64) * 512);
    ready = o;      o = align_up(o + (decode ? 4 * ((size_t)dtiles + 1) : 0));   // + plan flag
    xb_perm = o;    o = align_up(o + (w16 ? 2 * (size_t)Rt * H : 0));
    hb = o;         o = align_up(o + (w16 ? 2 * (size_t)Rt * I : 0));
    xq8 = o;        o = align_up(o + (mx ? (size_t)T * H + (size_t)T * H / 32 : 0));
    hq8 = o;        o = align_up(o + (mx ? (size_t)Rt * I + (size_t)Rt * I / 32 : 0));
    total = o;
  }
};

// Header words inside a workspace.
struct WsHeader {
  int32_t status;     // device status word
  float ts;           // activation tensor scale
  uint32_t counter;   // last-block counter of the amax reduction (returns to 0 after each call)
  uint32_t pad[61];
};

// ---- launchers (return a cudaError_t) ----
cudaError_t launch_act_quant(const void* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                             float* ts, WsHeader* hdr, uint32_t* partials, float* zero_buf,
                             int64_t zero_floats, cudaStream_t s);

// The two halves of launch_act_quant for batches that are planned before they are encoded:
// max |x| -> tensor scale (and the accumulator zeroing), then the encode into token order
// (codes / sf; null: skipped) and into every expert row of each token (xq_perm, xsf_tiles).
// With ts_in (already quantised input) the first half only zeroes the accumulator and copies
// *ts_in into the header.
cudaError_t launch_act_amax(const void* x, int64_t rows, int64_t cols, float* ts, WsHeader* hdr,
                            uint32_t* partials, float* zero_buf, int64_t zero_floats,
                            cudaStream_t s, const float* ts_in);
cudaError_t launch_act_encode_perm(const void* x, int T, int H, int k, int E, int shared, int Rt,
                                   const float* ts, const int32_t* ids, const int32_t* inv,
                                   const int32_t* offsets, const int32_t* tile_start,
                                   uint8_t* codes, uint8_t* sf, uint8_t* xq_perm,
                                   uint8_t* xsf_tiles, int32_t* status, cudaStream_t s);

// RMSNorm (FP32) of x [rows, cols] BF16 with gamma [cols] BF16, then NVFP4 with the tensor scale
// of the normalised values; each row's 1/rms also to rrms (may be null); scratch: 4 + rows words.
cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t rows,
                                 int64_t cols, uint8_t* codes, uint8_t* sf, float* ts,
                                 float* rrms, uint32_t* scratch, int32_t* status, cudaStream_t s);

cudaError_t launch_weight_quant(const moe_config& c, const WeightLayout& L, const void* wg,
                                const void* wu, const void* wd, const void* sg, const void* su,
                                const void* sd, uint8_t* wbuf, cudaStream_t s);

cudaError_t launch_weight_export(const moe_config& c, const WeightLayout& L, const uint8_t* wbuf,
                                 int expert_slot, int matrix, uint8_t* codes, uint8_t* sf, float* ts,
                                 cudaStream_t s);

struct PlanArgs {
  const float* logits;
  int T, E, k;
  int shared_rows;        // T when a shared-expert segment follows the routed rows, else 0
  int32_t* ids;           // [T*k]
  float* w;               // [T*k]
  int32_t* counts;        // [E] (may be null)
  int32_t* offsets;       // [E+1 (+1 with shared rows)] segment row offsets
  int32_t* tile_start;    // [E+1 (+1)] m-tile prefix (may be null)
  int32_t* perm_src;      // [R + shared_rows]
  float* perm_w;          // [R + shared_rows] (may be null)
  int32_t* inv;           // [T*k]
  int32_t* perm_seg;      // [R + shared_rows] expert (segment) of each permuted row (may be null)
  int32_t* hist;          // [nchunks*E + 1 + E] scratch: histograms, scan block count, totals
  int32_t* base;          // [nchunks*E] scratch
  int32_t* status;
  int sqrtsp;             // 1: the variant router (sqrt-softplus scores + selection bias)
  const float* bias;      // [E] selection bias of the variant router (may be null)
};
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s);

struct GemmArgs {
  // A operand: codes [*, K/2] and scales [*, K/16] rows; tile row r of segment s reads row
  // a_gather[m0 + r] (or m0 + r when a_gather is null).
  const uint8_t* a_codes;
  const uint8_t* a_sf;
  const int32_t* a_gather;
  // B operand: expert s's packed blocks start at b_tiles + s*b_per_seg ([N/128][K/256] blocks
  // of kTileBlockBytes, see WeightLayout).
  const uint8_t* b_tiles;
  size_t b_per_seg;
  const float* w_ts;      // [nseg][4] tensor scales
  const int32_t* seg_off; // [nseg+1]
  const int32_t* tile_start;  // [nseg+1]
  int nseg;
  int N, K;
  // epilogue
  int mode;               // 0: SwiGLU + requant (GEMM1); 1: down projection, router-weighted
                          // reduction into yacc; 2: down projection, router-weighted row stored
                          // to obuf (row = permuted row)
  const float* ts_a;      // device scalar (mode 0)
  float ts_h;
  uint8_t* hq;            // mode 0 out [rows, N/4]   (h has N/2 features)
  uint8_t* hsf;           // mode 0 out [rows, N/32]
  const int32_t* perm_src;  // mode 1: token of each permuted row
  const float* perm_w;      // modes 1 and 2: router weight of each permuted row
  float* yacc;              // mode 1 out [T, N]
  float* obuf;              // mode 2 out [rows, N]
  int act;                  // mode 0, the activation (kAct* in common.cuh): SwiGLU, clamped
                            // SwiGLU, ReLU2 (non-gated: N = I columns, no gate), SwiGLU-OAI
  float swiglu_limit;
  float swiglu_alpha;
  int32_t* status;
  int max_ctas;
  // bounds used to reject malformed plan data instead of touching memory outside the buffers
  int a_rows;             // rows of the A operand (tokens for GEMM1, permuted rows for GEMM2)
  int out_rows;           // rows of hq / hsf (mode 0) or of the permuted space (mode 1)
  int y_rows;             // rows of yacc (mode 1)
  int max_items;          // upper bound of m-tiles x n-tiles
  // decode kernel only: token rows are contiguous per expert (a_codes in permuted order, read
  // through a tensor map), their scales pre-arranged per expert tile, and GEMM1 also writes the
  // scales of h in that arrangement for GEMM2
  const uint8_t* a_sf_tiles;  // [tiles][K/64][512]
  uint8_t* hsf_tiles;         // mode 0 out [tiles][(N/2)/64][512]
};
cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s);

// The W4A16 / W4A8 layers' grouped GEMM on kind::f16 tensor cores (gemm_w16.cu; weights decoded
// to BF16 in shared memory): 256 expert-ordered token rows x 128 weight rows per tile, or, swapped,
// 128 weight rows x 16 token rows.  Its tile table is built in the kernel from seg_off.
struct GemmW16Args {
  const void* a_rows;         // A operand: BF16 rows [out_rows, K] in expert order
  const uint8_t* b_tiles;     // packed NVFP4 weight blocks (WeightLayout), expert s at s*b_per_seg
  size_t b_per_seg;
  const float* w_ts;          // [nseg][4] tensor scales
  const int32_t* seg_off;     // [nseg+1]
  int nseg;
  int N, K;
  int mode;                   // 0: activation, h to BF16 rows (hb [out_rows, I]); 1: router-
                              // weighted FP32 reduction into yacc [y_rows, N]
  int act;                    // kAct* (mode 0)
  float swiglu_limit, swiglu_alpha;
  uint8_t* hb;                // mode 0 out, BF16 [out_rows, I]
  int mx;                     // W4A8: MXFP4 weight blocks (E8M0 scales, no tensor scale) and h
                              // requantised to MXFP8 (codes to hq8, scales to hsf8; hb decoded)
  uint8_t* hq8;               // mode 0, mx: E4M3 codes [out_rows, I]
  uint8_t* hsf8;              // mode 0, mx: E8M0 scales [out_rows, I/32]
  const int32_t* perm_src;    // mode 1: token of each permuted row
  const float* perm_w;        // mode 1: router weight of each permuted row
  float* yacc;                // mode 1 out [y_rows, N]
  int out_rows, y_rows, max_items;
  int32_t* status;
  // decode-sized batches: the decoded weights are the MMA's 128-row A operand and tiles of
  // kDecodeTileRows expert-ordered token rows its N; max_items counts the tiles of either layout
  // x N/128
  int swap;
};
cudaError_t launch_grouped_gemm_w16(const GemmW16Args& a, cudaStream_t s);

// The W4A8 layer's activation quantiser: MXFP8 codes [T, H] and E8M0 scales [T, H/32] in token
// order, and the decoded BF16 values in every expert row of each token (xb_perm [Rt, H]).
cudaError_t launch_act_mx_encode_perm(const void* x, int T, int H, int k, int shared, int Rt,
                                      const int32_t* inv, uint8_t* codes, uint8_t* sf,
                                      void* xb_perm, int32_t* status, cudaStream_t s);

// Copies BF16 token rows into expert order: row p of xb_perm is row perm_src[p] of x [T, H].
cudaError_t launch_permute_rows_bf16(const void* x, int T, int H, int Rt, const int32_t* perm_src,
                                     void* xb_perm, int32_t* status, cudaStream_t s);

// Decode-sized batches (T <= kDecodeMaxRows): both grouped GEMMs in one persistent launch
// (gemm_decode.cu), weights as the MMA's M operand and tiles of kDecodeTileRows token rows of one
// expert as N.  Every CTA first takes its GEMM1 items (tile, 128-row tile of the interleaved
// gate/up weights), then its GEMM2 items (tile, 128-row tile of the down weights); a GEMM2 item
// reads the tile's h rows only once all GEMM1 epilogue warps of that tile have published them in
// `ready`.
struct DecodeGemmArgs {
  GemmArgs g1;          // gate/up projection, SwiGLU + requantisation (mode 0)
  GemmArgs g2;          // down projection, router-weighted rows stored to obuf (mode 2)
  int32_t* ready;       // [tiles] finished GEMM1 epilogue warps per tile; zeroed by the decode
                        // prologue of the same call
  const int32_t* plan_flag;   // set by the decode prologue once the plan is in global memory
};
cudaError_t launch_grouped_gemm_decode(const DecodeGemmArgs& a, cudaStream_t s);
// 2-D tensor map encoder of the driver, fetched through the runtime (no libcuda link).
bool tensor_map_available();

cudaError_t launch_finalize(const float* yacc, void* y, int64_t n, cudaStream_t s);

// Copies quantised activation rows into expert (permuted) order and scatters their scale words
// into the GEMM's tile arrangement: row p takes token perm_src[p]; its tile is
// tile_start[e] + (p - offsets[e]) / 128 for its expert e = perm_seg[p].
cudaError_t launch_permute_rows(const uint8_t* xq, const uint8_t* xsf, int T, int H, int Rt,
                                int E, const int32_t* perm_src, const int32_t* perm_seg,
                                const int32_t* offsets, const int32_t* tile_start,
                                uint8_t* xq_perm, uint8_t* xsf_tiles, int32_t* status,
                                cudaStream_t s);
cudaError_t launch_finalize_gather(const float* o, const int32_t* inv, int T, int k, int H,
                                   int shared, void* y, cudaStream_t s,
                                   int32_t* plan_flag = nullptr);

struct PrologueArgs {
  const void* x;           // [T, H] BF16
  int T, H;
  int32_t* status;
  float* ts;
  uint8_t* xq;             // [T, H/2]
  uint8_t* xsf;            // [T, H/16]
  const float* logits;     // [T, E]
  int E, k, shared_rows;
  int32_t *ids, *counts, *offsets, *tile_start, *perm_src, *inv, *perm_seg;
  float *w, *perm_w;
  int sqrtsp;              // the variant router (see PlanArgs)
  const float* bias;
  const float* in_ts;      // non-null: x is already quantised (its codes are permuted later);
                           // only this tensor scale is copied to ts, nothing is encoded
};
cudaError_t launch_prologue_small(const PrologueArgs& a, cudaStream_t s);

// Decode batches: the prologue as a cluster that also writes the activations in expert order.
constexpr int kDecodeProCtas = 8;
struct DecodePrologueArgs {
  const void* x;           // [T, H] BF16
  int T, H;
  int32_t* status;
  float* ts;
  uint8_t* xq;             // [T, H/2]  token order (null: not written)
  uint8_t* xsf;            // [T, H/16]
  uint8_t* xq_perm;        // [Rt, H/2] permuted (expert) order
  uint8_t* xsf_tiles;      // [tiles][H/64][512] token-operand scale arrangement
  const float* logits;     // [T, E]
  int E, k, shared_rows;
  int32_t *ids, *counts, *offsets, *tile_start, *perm_src, *inv, *perm_seg;
  float *w, *perm_w;
  int sqrtsp;              // the variant router (see PlanArgs)
  const float* bias;
  int32_t* ready;          // [nready] readiness counts of the decode GEMM, zeroed here
  int nready;
  int32_t* plan_flag;      // 0 before this kernel lets the GEMM launch, 1 once the plan is written
  // already quantised input (all null for BF16 x): codes [T, H/2], scales [T, H/16] and the
  // tensor scale, copied into expert order as they are (xq / xsf are then not written)
  const uint8_t* in_xq;
  const uint8_t* in_xsf;
  const float* in_ts;
  int no_plan_flag;        // test hook (MOE_INJECT_NO_PLAN_FLAG): never raise plan_flag
};
cudaError_t launch_decode_prologue(const DecodePrologueArgs& a, cudaStream_t s);

int num_sms();

// Launches `kernel` with the programmatic-stream-serialization attribute (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace nvfp4moe
