// Internal declarations of the NVFP4 MoE library: buffer layouts and kernel launchers.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nvfp4_moe.h"

namespace nvfp4moe {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// GEMM tiling shared by the host and the kernels.
constexpr int kBM = 128;       // permuted rows per tile (MMA M)
constexpr int kBN = 128;       // output columns per tile (MMA N)
constexpr int kBK = 256;       // FP4 elements of K per pipeline stage (128 bytes per row)
constexpr int kMmaK = 64;      // K of one block-scaled FP4 MMA

// Router chunking: tokens per chunk (one router block and one scatter block each).
inline int plan_tokens_per_chunk(int k) { return k <= 16 ? 64 : 32; }

// Private layout of the packed-weight buffer.
//   w13 codes [Et][2I][H/2]: row 32b+i is gate row 16b+i for i < 16, else up row 16b+i-16.
//   w13 sf    [Et][2I/128][H/64][512 B]: per 128-row group and 64-wide K chunk, one 512-byte
//             block with byte (n%32)*16 + ((n%128)/32)*4 + (k/16)%4 for row n, column k.
//   w2 codes  [Et][H][I/2];  w2 sf [Et][H/128][I/64][512 B] (same arrangement).
//   ts        [Et][4] FP32: gate, up, down tensor scales (the 4th is padding).
// Et = E + 1 with a shared expert, which is stored last.
struct WeightLayout {
  int E, Et, H, I;
  size_t w13_codes, w13_sf, w2_codes, w2_sf, ts, total;
  size_t w13_codes_per_e, w13_sf_per_e, w2_codes_per_e, w2_sf_per_e;
  explicit WeightLayout(const moe_config& c) {
    E = c.num_experts;
    Et = E + (c.shared_inter > 0 ? 1 : 0);
    H = c.hidden;
    I = c.inter;
    w13_codes_per_e = (size_t)2 * I * H / 2;
    w13_sf_per_e = (size_t)2 * I * H / 16;
    w2_codes_per_e = (size_t)H * I / 2;
    w2_sf_per_e = (size_t)H * I / 16;
    size_t o = 0;
    w13_codes = o; o = align_up(o + w13_codes_per_e * Et);
    w13_sf = o;    o = align_up(o + w13_sf_per_e * Et);
    w2_codes = o;  o = align_up(o + w2_codes_per_e * Et);
    w2_sf = o;     o = align_up(o + w2_sf_per_e * Et);
    ts = o;        o = align_up(o + sizeof(float) * 4 * Et);
    total = o;
  }
};

// Workspace of moe_run for T tokens.  Offset 0 holds the device status word.
struct RunLayout {
  size_t hdr, amax_part, ids, w, hist, base, seg_off, tile_start, perm_src, perm_w, inv, xq, xsf,
      hq, hsf, yacc, total;
  int T, R, Rt, nseg, nchunks, tpc;
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
    hist = o;       o = align_up(o + 4 * (size_t)nchunks * E);
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
    yacc = o;       o = align_up(o + 4 * (size_t)T * H);
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
  int32_t* hist;          // [nchunks*E] scratch
  int32_t* base;          // [nchunks*E] scratch
  int32_t* status;
};
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s);

struct GemmArgs {
  // A operand: codes [*, K/2] and scales [*, K/16] rows; tile row r of segment s reads row
  // a_gather[m0 + r] (or m0 + r when a_gather is null).
  const uint8_t* a_codes;
  const uint8_t* a_sf;
  const int32_t* a_gather;
  // B operand: expert s owns rows [s*N, (s+1)*N) of the codes tensor map and the packed scale
  // block b_sf + s*b_sf_per_seg.
  const uint8_t* b_sf;
  size_t b_sf_per_seg;
  const float* w_ts;      // [nseg][4] tensor scales
  const int32_t* seg_off; // [nseg+1]
  const int32_t* tile_start;  // [nseg+1]
  int nseg;
  int N, K;
  // epilogue
  int mode;               // 0: SwiGLU + requant (GEMM1), 1: down projection + weighted combine
  const float* ts_a;      // device scalar (mode 0)
  float ts_h;
  uint8_t* hq;            // mode 0 out [rows, N/4]   (h has N/2 features)
  uint8_t* hsf;           // mode 0 out [rows, N/32]
  const int32_t* perm_src;  // mode 1
  const float* perm_w;      // mode 1
  float* yacc;              // mode 1 out [T, N]
  int32_t* status;
  int max_ctas;
  // bounds used to reject malformed plan data instead of touching memory outside the buffers
  int a_rows;             // rows of the A operand (tokens for GEMM1, permuted rows for GEMM2)
  int out_rows;           // rows of hq / hsf (mode 0) or of the permuted space (mode 1)
  int y_rows;             // rows of yacc (mode 1)
  int max_items;          // upper bound of m-tiles x n-tiles
};
cudaError_t launch_grouped_gemm(const GemmArgs& a, const uint8_t* b_codes, int b_rows_total,
                                cudaStream_t s);

cudaError_t launch_finalize(const float* yacc, void* y, int64_t n, cudaStream_t s);

int num_sms();

}  // namespace nvfp4moe
