// C ABI of the NVFP4 MoE library: argument checks, workspace carving and the launch sequence.
// Nothing here allocates device memory or reads device values back to the host (the single
// exception is moe_last_device_status, which exists to do exactly that).
#include <algorithm>
#include <cmath>
#include <tuple>

#include "internal.h"

using namespace nvfp4moe;

namespace {

inline cudaStream_t to_cuda(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace behind the layer's own when a width is padded (pc = padded_config(c)): x, or its
// codes and scales, in rows of the padded width; then the BF16 output rows before their copy
// into y.
size_t pad_bytes(const moe_config& c, const moe_config& pc, int32_t T) {
  if (!needs_padding(c)) return 0;
  return 2 * align_up((size_t)T * pc.hidden * 2);
}

int check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const uint32_t acts = MOE_FLAG_SWIGLU_CLAMP | MOE_FLAG_ACT_RELU2 | MOE_FLAG_ACT_SWIGLU_OAI;
  if ((c->flags & ~(MOE_FLAG_ROUTER_SQRTSOFTPLUS | acts | MOE_FLAG_ACT_BF16 |
                    MOE_FLAG_ACT_MXFP8)) != 0u)
    return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_ACT_BF16) && (c->flags & MOE_FLAG_ACT_MXFP8)) return MOE_ERR_INVALID_ARG;
  const uint32_t act = c->flags & acts;
  if (act & (act - 1u)) return MOE_ERR_INVALID_ARG;   // at most one activation
  if ((act & (MOE_FLAG_SWIGLU_CLAMP | MOE_FLAG_ACT_SWIGLU_OAI)) &&
      !(std::isfinite(c->swiglu_limit) && c->swiglu_limit >= 0.0f))
    return MOE_ERR_INVALID_ARG;
  if ((act & MOE_FLAG_ACT_SWIGLU_OAI) && !std::isfinite(c->swiglu_alpha)) return MOE_ERR_INVALID_ARG;
  if (c->num_experts < 1 || c->top_k < 1 || c->hidden <= 0 || c->inter <= 0 || c->max_tokens < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->num_experts) return MOE_ERR_INVALID_ARG;
  if (!(std::isfinite(c->h_tensor_scale) && c->h_tensor_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (c->num_experts > 1024 || c->top_k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden % 32 != 0 || c->inter % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden > (1 << 20) || c->inter > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->shared_inter < 0) return MOE_ERR_INVALID_ARG;
  if (c->shared_inter % 32 != 0 || c->shared_inter > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace or buffer too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite input maximum";
    case MOE_ERR_UNIMPLEMENTED: return "not implemented";
    default: return "unknown status";
  }
}

int moe_config_check(const moe_config* cfg) { return check_cfg(cfg); }

size_t moe_weights_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return WeightLayout(padded_config(*cfg)).total;
}

int moe_quantize_weights(const moe_config* cfg, const void* w_gate, const void* w_up,
                         const void* w_down, const void* s_gate, const void* s_up,
                         const void* s_down, void* wbuf, size_t wbuf_bytes, moe_stream_t stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  const bool gated = gated_experts(*cfg);
  if (!gated) {   // non-gated experts: the gate matrices are not read
    w_gate = nullptr;
    s_gate = nullptr;
  }
  if ((gated && !w_gate) || !w_up || !w_down || !wbuf) return MOE_ERR_INVALID_ARG;
  if (cfg->shared_inter > 0 && ((gated && !s_gate) || !s_up || !s_down)) return MOE_ERR_INVALID_ARG;
  for (const void* p : {w_gate, w_up, w_down})
    if (p && !aligned(p, 16)) return MOE_ERR_INVALID_ARG;
  if (cfg->shared_inter > 0)
    for (const void* p : {s_gate, s_up, s_down})
      if (p && !aligned(p, 16)) return MOE_ERR_INVALID_ARG;
  if (!aligned(wbuf, kAlign)) return MOE_ERR_INVALID_ARG;
  const WeightLayout L(padded_config(*cfg));
  if (wbuf_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = to_cuda(stream);
  uint8_t* wb = static_cast<uint8_t*>(wbuf);
  if (cudaMemsetAsync(wb + L.bias, 0, sizeof(float) * L.E, s) != cudaSuccess) return MOE_ERR_CUDA;
  // padded widths: the packed blocks' padding rows and columns are zero codes and zero scales
  if (needs_padding(*cfg) && cudaMemsetAsync(wb + L.w13, 0, L.ts - L.w13, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(launch_weight_quant(*cfg, L, w_gate, w_up, w_down, s_gate, s_up, s_down, wb, s));
}

int moe_set_router_bias(const moe_config* cfg, void* wbuf, const float* bias, moe_stream_t stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!wbuf || !bias || !aligned(wbuf, kAlign)) return MOE_ERR_INVALID_ARG;
  const WeightLayout L(padded_config(*cfg));
  return cuda_status(cudaMemcpyAsync(static_cast<uint8_t*>(wbuf) + L.bias, bias,
                                     sizeof(float) * L.E, cudaMemcpyDeviceToDevice,
                                     to_cuda(stream)));
}

int moe_weights_export(const moe_config* cfg, const void* wbuf, int32_t expert, int32_t matrix,
                       uint8_t* codes, uint8_t* sf, float* ts, moe_stream_t stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!wbuf || !codes || !sf || !ts) return MOE_ERR_INVALID_ARG;
  if (matrix < 0 || matrix > 2) return MOE_ERR_INVALID_ARG;
  if (matrix == 0 && !gated_experts(*cfg)) return MOE_ERR_INVALID_ARG;   // no gate matrix
  // (sf receives [N, K/16] E4M3 scales, or [N, K/32] E8M0 scales for MXFP4 weights)
  int slot;
  if (expert == -1) {
    if (cfg->shared_inter <= 0) return MOE_ERR_INVALID_ARG;
    slot = cfg->num_experts;
  } else if (expert >= 0 && expert < cfg->num_experts) {
    slot = expert;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  if (!aligned(codes, 8)) return MOE_ERR_INVALID_ARG;
  const WeightLayout L(padded_config(*cfg));
  return cuda_status(launch_weight_export(*cfg, L, static_cast<const uint8_t*>(wbuf), slot, matrix,
                                          codes, sf, ts, to_cuda(stream)));
}

size_t moe_act_workspace_size(int64_t rows, int64_t cols) {
  (void)rows;
  (void)cols;
  return 256 + 4 * 1024;
}

int moe_quantize_act(const void* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                     float* ts, void* workspace, size_t ws_bytes, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < moe_act_workspace_size(rows, cols)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 16)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !sf || !ts) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(ts, 4)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = to_cuda(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t* partials = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + 256);
  return cuda_status(launch_act_quant(x, rows, cols, codes, sf, ts, hdr, partials, nullptr, 0, s));
}

size_t moe_rmsnorm_workspace_size(int64_t rows) {
  if (rows < 0) return 0;
  return 256 + align_up(4 * (4 + (size_t)rows));
}

int moe_rmsnorm_quantize_act(const void* x, const void* gamma, float eps, int64_t rows,
                             int64_t cols, uint8_t* codes, uint8_t* sf, float* ts, float* rrms,
                             void* workspace, size_t ws_bytes, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || !(std::isfinite(eps) && eps >= 0.0f))
    return MOE_ERR_INVALID_ARG;
  if (cols > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || ws_bytes < moe_rmsnorm_workspace_size(rows)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 16)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !gamma || !codes || !sf || !ts) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(codes, 8) || !aligned(ts, 4))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = to_cuda(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t* scratch = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + 256);
  if (rrms && !aligned(rrms, 4)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm_quant(x, gamma, eps, rows, cols, codes, sf, ts, rrms, scratch,
                                          &hdr->status, s));
}

size_t moe_plan_workspace_size(int32_t T, int32_t E, int32_t k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  const int tpc = plan_tokens_per_chunk(k);
  const size_t nchunks = ((size_t)T + tpc - 1) / tpc;
  return 256 + align_up(4 * (nchunks * E + 1 + E)) + align_up(4 * nchunks * E);
}

int moe_plan(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
             float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv,
             void* workspace, size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < moe_plan_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = to_cuda(stream);
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!logits || !topk_ids || !topk_w || !perm_src || !inv) return MOE_ERR_INVALID_ARG;
  const int tpc = plan_tokens_per_chunk(k);
  const size_t nchunks = ((size_t)T + tpc - 1) / tpc;
  uint8_t* w8 = static_cast<uint8_t*>(workspace);
  PlanArgs a{};
  a.logits = logits;
  a.T = T;
  a.E = E;
  a.k = k;
  a.shared_rows = 0;
  a.ids = topk_ids;
  a.w = topk_w;
  a.counts = counts;
  a.offsets = offsets;
  a.tile_start = nullptr;
  a.perm_src = perm_src;
  a.perm_w = nullptr;
  a.inv = inv;
  a.hist = reinterpret_cast<int32_t*>(w8 + 256);
  a.base = reinterpret_cast<int32_t*>(w8 + 256 + align_up(4 * (nchunks * E + 1 + E)));
  a.status = reinterpret_cast<int32_t*>(w8);
  return cuda_status(launch_plan(a, s));
}

size_t moe_workspace_size(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 0) return 0;
  const moe_config pc = padded_config(*cfg);
  return RunLayout(pc, T).total + pad_bytes(*cfg, pc, T);
}

int moe_run_kernel_count(const moe_config* cfg, int32_t T) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return 0;
  const RunLayout L(padded_config(*cfg), T);
  if (L.decode) return 3;     // cluster prologue, both grouped GEMMs, row sum
  if (L.small) return 5;      // one-block prologue, permute, GEMM1, GEMM2, row sum
  // accumulator zeroing (+ amax), router/plan (1 or 3), encode (or, W4A16, the BF16 rows) into
  // expert order, GEMM1, GEMM2, BF16 conversion
  return 1 + ((int64_t)T * cfg->top_k <= kSmallPlanRows ? 1 : 3) + 4;
}

}  // extern "C"

namespace {

// The layer for BF16 input x (qx == nullptr) or for already quantised input (qx: codes
// [T, H/2], qsf: scales [T, H/16], qts: device tensor scale; x unused), at widths that are
// multiples of 256.  Hl, Il: the caller's widths (equal to cfg's unless run_layer padded them),
// used for the debug copies.
int run_core(const moe_config* cfg, int Hl, int Il, const void* wbuf, const void* x,
             const uint8_t* qx, const uint8_t* qsf, const float* qts, const float* logits,
             int32_t T, int32_t k, void* y, void* workspace, size_t ws_bytes,
             moe_stream_t stream, const moe_debug* debug) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0 || k != cfg->top_k) return MOE_ERR_INVALID_ARG;
  if (cfg->max_tokens > 0 && T > cfg->max_tokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)T * (cfg->top_k + 1) > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  const RunLayout L(*cfg, T);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const bool quantised = qx != nullptr || qsf != nullptr || qts != nullptr;
  if (quantised && L.w16) return MOE_ERR_INVALID_ARG;   // a W4A16 layer takes BF16 input
  if (!wbuf || !logits || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(wbuf, kAlign) || !aligned(y, 8)) return MOE_ERR_INVALID_ARG;
  if (quantised) {
    if (!qx || !qsf || !qts) return MOE_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(qsf, 4) || !aligned(qts, 4)) return MOE_ERR_INVALID_ARG;
  } else if (!x || !aligned(x, 16)) {
    return MOE_ERR_INVALID_ARG;
  }

  cudaStream_t s = to_cuda(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* wb = static_cast<const uint8_t*>(wbuf);
  const WeightLayout W(*cfg);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.hdr);
  const int E = cfg->num_experts, H = cfg->hidden, I = cfg->inter;
  const int shared = cfg->shared_inter > 0 ? 1 : 0;
  const int sqrtsp = (cfg->flags & MOE_FLAG_ROUTER_SQRTSOFTPLUS) ? 1 : 0;
  const float* rbias = reinterpret_cast<const float*>(wb + W.bias);

  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };

  cudaEvent_t* ev = (debug && debug->stage_events) ? reinterpret_cast<cudaEvent_t*>(debug->stage_events)
                                                    : nullptr;
  // inside a stream capture the events must become record nodes of the graph
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (ev && cudaStreamIsCapturing(s, &capture) != cudaSuccess) return MOE_ERR_CUDA;
  auto mark = [&](int i) {
    if (!ev) return cudaSuccess;
    return capture == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev[i], s, cudaEventRecordExternal)
               : cudaEventRecord(ev[i], s);
  };

  cudaError_t e = mark(0);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  if (L.w16) {
    // W4A16: accumulator zeroing, router + plan, BF16 rows into expert order, both GEMMs on the
    // BF16 tensor cores (weights decoded in shared memory), BF16 output
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_act_amax(x, 0, H, nullptr, hdr, reinterpret_cast<uint32_t*>(ws + L.amax_part),
                        f32(L.yacc), (int64_t)T * H, s, nullptr);
    if (e == cudaSuccess) e = mark(1);
    PlanArgs pa{};
    pa.logits = logits;
    pa.T = T;
    pa.E = E;
    pa.k = k;
    pa.shared_rows = shared ? T : 0;
    pa.ids = i32(L.ids);
    pa.w = f32(L.w);
    pa.counts = debug ? debug->counts : nullptr;
    pa.offsets = i32(L.seg_off);
    pa.tile_start = i32(L.tile_start);
    pa.perm_src = i32(L.perm_src);
    pa.perm_w = f32(L.perm_w);
    pa.inv = i32(L.inv);
    pa.perm_seg = i32(L.perm_seg);
    pa.hist = i32(L.hist);
    pa.base = i32(L.base);
    pa.status = &hdr->status;
    pa.sqrtsp = sqrtsp;
    pa.bias = rbias;
    if (e == cudaSuccess) e = launch_plan(pa, s);
    if (e == cudaSuccess) e = mark(2);
    if (e == cudaSuccess)
      e = L.mx ? launch_act_mx_encode_perm(x, T, H, k, shared, L.Rt, i32(L.inv), ws + L.xq8,
                                           ws + L.xq8 + (size_t)T * H, ws + L.xb_perm,
                                           &hdr->status, s)
               : launch_permute_rows_bf16(x, T, H, L.Rt, i32(L.perm_src), ws + L.xb_perm,
                                          &hdr->status, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const int nseg = E + shared;
    // decode-sized batches: weights as the MMA's M operand, kDecodeTileRows token rows as its N;
    // otherwise 256-row token tiles (two 128-row MMA operands sharing each decoded weight tile)
    const bool swap = T <= kDecodeMaxRows;
    const int tr = swap ? kDecodeTileRows : 2 * kBM;
    const int64_t mtiles = ((int64_t)L.Rt + (int64_t)nseg * (tr - 1)) / tr;
    GemmW16Args g{};
    g.a_rows = ws + L.xb_perm;
    g.b_tiles = wb + W.w13;
    g.b_per_seg = W.w13_per_e;
    g.w_ts = reinterpret_cast<const float*>(wb + W.ts);
    g.seg_off = i32(L.seg_off);
    g.nseg = nseg;
    g.N = gemm1_rows(*cfg);
    g.K = H;
    g.mode = 0;
    g.act = (cfg->flags & MOE_FLAG_SWIGLU_CLAMP) ? kActSwigluClamp
            : (cfg->flags & MOE_FLAG_ACT_RELU2)   ? kActRelu2
            : (cfg->flags & MOE_FLAG_ACT_SWIGLU_OAI) ? kActSwigluOai
                                                    : kActSwiglu;
    g.swiglu_limit = cfg->swiglu_limit;
    g.swiglu_alpha = cfg->swiglu_alpha;
    g.hb = ws + L.hb;
    g.mx = L.mx ? 1 : 0;
    g.hq8 = ws + L.hq8;
    g.hsf8 = ws + L.hq8 + (size_t)L.Rt * I;
    g.out_rows = L.Rt;
    g.y_rows = T;
    g.max_items = (int)std::min<int64_t>(mtiles * (g.N / kBN), INT32_MAX);
    g.status = &hdr->status;
    g.swap = swap ? 1 : 0;
    e = launch_grouped_gemm_w16(g, s);
    if (e == cudaSuccess) e = mark(3);
    GemmW16Args g2 = g;
    g2.a_rows = ws + L.hb;
    g2.b_tiles = wb + W.w2;
    g2.b_per_seg = W.w2_per_e;
    g2.N = H;
    g2.K = I;
    g2.mode = 1;
    g2.perm_src = i32(L.perm_src);
    g2.perm_w = f32(L.perm_w);
    g2.yacc = f32(L.yacc);
    g2.max_items = (int)std::min<int64_t>(mtiles * (g2.N / kBN), INT32_MAX);
    if (e == cudaSuccess) e = launch_grouped_gemm_w16(g2, s);
    if (e == cudaSuccess) e = mark(4);
    if (e == cudaSuccess) e = launch_finalize(f32(L.yacc), y, (int64_t)T * H, s);
    if (e == cudaSuccess) e = mark(5);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (debug) {
      auto cp = [&](void* dst, size_t off, size_t bytes) {
        if (dst && e == cudaSuccess)
          e = cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToDevice, s);
      };
      // rows of the caller's width out of rows of the layer's width
      auto cp2 = [&](void* dst, size_t off, size_t rows, size_t width, size_t pitch) {
        if (dst && e == cudaSuccess && rows > 0)
          e = cudaMemcpy2DAsync(dst, width, ws + off, pitch, width, rows,
                                cudaMemcpyDeviceToDevice, s);
      };
      const size_t R = (size_t)L.R, Rt = (size_t)L.Rt;
      cp(debug->topk_ids, L.ids, 4 * R);
      cp(debug->topk_w, L.w, 4 * R);
      cp(debug->offsets, L.seg_off, 4 * (size_t)(E + 1));
      cp(debug->perm_src, L.perm_src, 4 * R);
      cp(debug->inv, L.inv, 4 * R);
      cp2(debug->hb, L.hb, Rt, (size_t)Il * 2, (size_t)I * 2);
      if (L.mx) {   // MXFP8 codes and E8M0 scales of x and h
        cp2(debug->xq, L.xq8, T, Hl, H);
        cp2(debug->xsf, L.xq8 + (size_t)T * H, T, Hl / 32, H / 32);
        cp2(debug->hq, L.hq8, Rt, Il, I);
        cp2(debug->hsf, L.hq8 + Rt * I, Rt, Il / 32, I / 32);
      }
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }

  if (L.decode) {
    // 1+2. a cluster: status reset, router and plan, activation quantiser in expert order
    DecodePrologueArgs pr{};
    pr.x = x;
    pr.T = T;
    pr.H = H;
    pr.status = &hdr->status;
    pr.ts = &hdr->ts;
    // token-order codes feed nothing on this path but the debug copies
    pr.xq = debug ? ws + L.xq : nullptr;
    pr.xsf = debug ? ws + L.xsf : nullptr;
    pr.xq_perm = ws + L.xq_perm;
    pr.xsf_tiles = ws + L.xsf_tiles;
    pr.logits = logits;
    pr.E = E;
    pr.k = k;
    pr.shared_rows = shared ? T : 0;
    pr.ids = i32(L.ids);
    pr.w = f32(L.w);
    pr.counts = debug ? debug->counts : nullptr;
    pr.offsets = i32(L.seg_off);
    pr.tile_start = i32(L.tile_start);
    pr.perm_src = i32(L.perm_src);
    pr.perm_w = f32(L.perm_w);
    pr.inv = i32(L.inv);
    pr.perm_seg = i32(L.perm_seg);
    pr.sqrtsp = sqrtsp;
    pr.bias = rbias;
    pr.ready = i32(L.ready);
    pr.nready = L.dtiles;
    pr.plan_flag = i32(L.ready) + L.dtiles;
    pr.in_xq = qx;
    pr.in_xsf = qsf;
    pr.in_ts = qts;
    pr.no_plan_flag = (debug && (debug->inject & MOE_INJECT_NO_PLAN_FLAG)) ? 1 : 0;
    e = launch_decode_prologue(pr, s);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = mark(2);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (L.small) {
    // 1+2. one block: status reset, activation quantiser, router and plan
    PrologueArgs pr{};
    pr.x = x;
    pr.T = T;
    pr.H = H;
    pr.status = &hdr->status;
    pr.ts = &hdr->ts;
    pr.xq = ws + L.xq;
    pr.xsf = ws + L.xsf;
    pr.logits = logits;
    pr.E = E;
    pr.k = k;
    pr.shared_rows = shared ? T : 0;
    pr.ids = i32(L.ids);
    pr.w = f32(L.w);
    pr.counts = debug ? debug->counts : nullptr;
    pr.offsets = i32(L.seg_off);
    pr.tile_start = i32(L.tile_start);
    pr.perm_src = i32(L.perm_src);
    pr.perm_w = f32(L.perm_w);
    pr.inv = i32(L.inv);
    pr.perm_seg = i32(L.perm_seg);
    pr.sqrtsp = sqrtsp;
    pr.bias = rbias;
    pr.in_ts = qts;
    e = launch_prologue_small(pr, s);
    if (e == cudaSuccess) e = mark(1);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else {
  e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // 1. activation tensor scale (and zero the FP32 output accumulator on the way); the encode
  //    follows the plan so that it can write every expert row directly
  e = launch_act_amax(x, T, H, nullptr, hdr, reinterpret_cast<uint32_t*>(ws + L.amax_part),
                      f32(L.yacc), (int64_t)T * H, s, qts);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // 2. router + plan
  PlanArgs pa{};
  pa.logits = logits;
  pa.T = T;
  pa.E = E;
  pa.k = k;
  pa.shared_rows = shared ? T : 0;
  pa.ids = i32(L.ids);
  pa.w = f32(L.w);
  pa.counts = debug ? debug->counts : nullptr;
  pa.offsets = i32(L.seg_off);
  pa.tile_start = i32(L.tile_start);
  pa.perm_src = i32(L.perm_src);
  pa.perm_w = f32(L.perm_w);
  pa.inv = i32(L.inv);
  pa.perm_seg = i32(L.perm_seg);
  pa.hist = i32(L.hist);
  pa.base = i32(L.base);
  pa.status = &hdr->status;
  pa.sqrtsp = sqrtsp;
  pa.bias = rbias;
  e = launch_plan(pa, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  const int nseg = E + shared;
  const int64_t max_mtiles = ((int64_t)L.Rt + (int64_t)nseg * (kBM - 1)) / kBM;
  // token-order codes and scales of the activations: the caller's (quantised input) or the
  // workspace copy the quantiser wrote
  const uint8_t* xq_tok = quantised ? qx : ws + L.xq;
  const uint8_t* xsf_tok = quantised ? qsf : ws + L.xsf;
  if ((L.small && !L.decode) || (quantised && !L.small)) {
    // activations (token order) into expert order
    e = launch_permute_rows(xq_tok, xsf_tok, T, H, L.Rt, E, i32(L.perm_src),
                            i32(L.perm_seg), i32(L.seg_off), i32(L.tile_start), ws + L.xq_perm,
                            ws + L.xsf_tiles, &hdr->status, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (!L.small) {
    // encode each block once into token order and into every expert row of its token
    // (the token-order codes feed nothing on this path but the debug copies)
    e = launch_act_encode_perm(x, T, H, k, E, shared, L.Rt, &hdr->ts, i32(L.ids), i32(L.inv),
                               i32(L.seg_off), i32(L.tile_start), debug ? ws + L.xq : nullptr,
                               debug ? ws + L.xsf : nullptr, ws + L.xq_perm, ws + L.xsf_tiles,
                               &hdr->status, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  // the router / plan stage ends once the activations are in expert order (the decode prologue
  // marked it already), so that GEMM1's stage times the GEMM alone
  if (!L.decode && mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  const float* w_ts = reinterpret_cast<const float*>(wb + W.ts);

  // 3. GEMM1 + SwiGLU + requantisation
  GemmArgs g{};
  g.a_codes = ws + L.xq;
  g.a_sf = ws + L.xsf;
  g.a_gather = i32(L.perm_src);
  g.b_tiles = wb + W.w13;
  g.b_per_seg = W.w13_per_e;
  g.w_ts = w_ts;
  g.seg_off = i32(L.seg_off);
  g.tile_start = i32(L.tile_start);
  g.nseg = nseg;
  g.N = gemm1_rows(*cfg);
  g.K = H;
  g.mode = 0;
  g.ts_a = &hdr->ts;
  g.ts_h = cfg->h_tensor_scale;
  g.hq = ws + L.hq;
  g.hsf = ws + L.hsf;
  g.status = &hdr->status;
  g.act = (cfg->flags & MOE_FLAG_SWIGLU_CLAMP) ? kActSwigluClamp
          : (cfg->flags & MOE_FLAG_ACT_RELU2)   ? kActRelu2
          : (cfg->flags & MOE_FLAG_ACT_SWIGLU_OAI) ? kActSwigluOai
                                                  : kActSwiglu;
  g.swiglu_limit = cfg->swiglu_limit;
  g.swiglu_alpha = cfg->swiglu_alpha;
  // decode-sized batches: tiles of kDecodeTileRows rows of one expert each
  const bool decode = L.decode;
  g.a_codes = ws + L.xq_perm;            // expert-ordered activations, read by TMA boxes
  g.a_sf_tiles = ws + L.xsf_tiles;
  g.hsf_tiles = ws + L.hsf_tiles;
  const int64_t item_rows = decode ? (int64_t)L.dtiles : max_mtiles;
  g.max_items = (int)std::min<int64_t>(item_rows * (g.N / kBN), INT32_MAX);
  g.max_ctas = g.max_items;
  g.a_rows = T;
  g.out_rows = L.Rt;
  g.y_rows = T;
  if (!decode) {
    e = launch_grouped_gemm(g, s);
    if (e == cudaSuccess) e = mark(3);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  // 4. GEMM2 (down projection) with the router-weighted accumulation into the token rows
  GemmArgs g2 = g;
  g2.a_codes = ws + L.hq;
  g2.a_sf = ws + L.hsf;
  g2.a_gather = nullptr;
  g2.a_sf_tiles = ws + L.hsf_tiles;
  g2.b_tiles = wb + W.w2;
  g2.b_per_seg = W.w2_per_e;
  g2.N = H;
  g2.K = I;
  g2.mode = L.small ? 2 : 1;
  g2.perm_src = i32(L.perm_src);
  g2.perm_w = f32(L.perm_w);
  g2.yacc = f32(L.yacc);
  g2.obuf = f32(L.obuf);
  g2.max_items = (int)std::min<int64_t>(item_rows * (g2.N / kBN), INT32_MAX);
  g2.max_ctas = g2.max_items;
  g2.a_rows = L.Rt;
  if (decode) {
    // both GEMMs in one persistent launch; its time is reported as GEMM1's stage
    DecodeGemmArgs dg{};
    dg.g1 = g;
    dg.g2 = g2;
    dg.ready = i32(L.ready);
    dg.plan_flag = i32(L.ready) + L.dtiles;
    e = launch_grouped_gemm_decode(dg, s);
    if (e == cudaSuccess) e = mark(3);
  } else {
    e = launch_grouped_gemm(g2, s);
  }
  if (e == cudaSuccess) e = mark(4);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // 5. BF16 output (small batches: sum each token's stored rows in slot order)
  e = L.small ? launch_finalize_gather(f32(L.obuf), i32(L.inv), T, k, H, shared, y, s,
                                       L.decode ? i32(L.ready) + L.dtiles : nullptr)
              : launch_finalize(f32(L.yacc), y, (int64_t)T * H, s);
  if (e == cudaSuccess) e = mark(5);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  if (debug) {
    auto cp = [&](void* dst, size_t off, size_t bytes) {
      if (dst && e == cudaSuccess) e = cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToDevice, s);
    };
    // rows of the caller's width out of rows of the layer's width
    auto cp2p = [&](void* dst, const void* src, size_t rows, size_t width, size_t pitch) {
      if (dst && e == cudaSuccess && rows > 0)
        e = cudaMemcpy2DAsync(dst, width, src, pitch, width, rows, cudaMemcpyDeviceToDevice, s);
    };
    auto cp2 = [&](void* dst, size_t off, size_t rows, size_t width, size_t pitch) {
      cp2p(dst, ws + off, rows, width, pitch);
    };
    const size_t R = (size_t)L.R, Rt = (size_t)L.Rt;
    cp(debug->topk_ids, L.ids, 4 * R);
    cp(debug->topk_w, L.w, 4 * R);
    cp(debug->offsets, L.seg_off, 4 * (size_t)(E + 1));
    cp(debug->perm_src, L.perm_src, 4 * R);
    cp(debug->inv, L.inv, 4 * R);
    if (quantised) {
      cp2p(debug->xq, qx, T, Hl / 2, H / 2);
      cp2p(debug->xsf, qsf, T, Hl / 16, H / 16);
    } else {
      cp2(debug->xq, L.xq, T, Hl / 2, H / 2);
      cp2(debug->xsf, L.xsf, T, Hl / 16, H / 16);
    }
    cp(debug->ts_a, L.hdr + offsetof(WsHeader, ts), 4);
    cp2(debug->hq, L.hq, Rt, Il / 2, I / 2);
    cp2(debug->hsf, L.hsf, Rt, Il / 16, I / 16);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// The layer at the caller's widths: directly when they are multiples of 256, otherwise through
// zero-padded copies of x (or of its codes and scales) and of the output rows in the workspace
// behind the layer's own (see padded_config).
int run_layer(const moe_config* cfg, const void* wbuf, const void* x, const uint8_t* qx,
              const uint8_t* qsf, const float* qts, const float* logits, int32_t T, int32_t k,
              void* y, void* workspace, size_t ws_bytes, moe_stream_t stream,
              const moe_debug* debug) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!needs_padding(*cfg))
    return run_core(cfg, cfg->hidden, cfg->inter, wbuf, x, qx, qsf, qts, logits, T, k, y,
                    workspace, ws_bytes, stream, debug);
  const int Il = h_width(*cfg);   // debug rows of h: the layer's widest intermediate
  if (T < 0 || k != cfg->top_k) return MOE_ERR_INVALID_ARG;
  if (cfg->max_tokens > 0 && T > cfg->max_tokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)T * (cfg->top_k + 1) > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  const moe_config pc = padded_config(*cfg);
  const size_t core = RunLayout(pc, T).total;
  if (ws_bytes < core + pad_bytes(*cfg, pc, T)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const bool quantised = qx != nullptr || qsf != nullptr || qts != nullptr;
  if (!y || !aligned(y, 8)) return MOE_ERR_INVALID_ARG;
  if (quantised) {
    if (!qx || !qsf || !qts) return MOE_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(qsf, 4) || !aligned(qts, 4)) return MOE_ERR_INVALID_ARG;
  } else if (!x || !aligned(x, 16)) {
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = to_cuda(stream);
  const size_t H = (size_t)cfg->hidden, Hp = (size_t)pc.hidden, rows = (size_t)T;
  uint8_t* xp = static_cast<uint8_t*>(workspace) + core;
  uint8_t* yp = xp + align_up(rows * Hp * 2);
  uint8_t* sfp = xp + align_up(rows * Hp / 2);   // quantised input: the scales after the codes
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (quantised) {
    if (!ok(cudaMemsetAsync(xp, 0, align_up(rows * Hp / 2) + rows * Hp / 16, s)) ||
        !ok(cudaMemcpy2DAsync(xp, Hp / 2, qx, H / 2, H / 2, rows, cudaMemcpyDeviceToDevice, s)) ||
        !ok(cudaMemcpy2DAsync(sfp, Hp / 16, qsf, H / 16, H / 16, rows, cudaMemcpyDeviceToDevice,
                              s)))
      return MOE_ERR_CUDA;
    st = run_core(&pc, cfg->hidden, Il, wbuf, nullptr, xp, sfp, qts, logits, T, k, yp,
                  workspace, core, stream, debug);
  } else {
    if (!ok(cudaMemsetAsync(xp, 0, rows * Hp * 2, s)) ||
        !ok(cudaMemcpy2DAsync(xp, Hp * 2, x, H * 2, H * 2, rows, cudaMemcpyDeviceToDevice, s)))
      return MOE_ERR_CUDA;
    st = run_core(&pc, cfg->hidden, Il, wbuf, xp, nullptr, nullptr, nullptr, logits, T, k, yp,
                  workspace, core, stream, debug);
  }
  if (st != MOE_OK) return st;
  return ok(cudaMemcpy2DAsync(y, H * 2, yp, Hp * 2, H * 2, rows, cudaMemcpyDeviceToDevice, s))
             ? MOE_OK
             : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

int moe_run(const moe_config* cfg, const void* wbuf, const void* x, const float* logits, int32_t T,
            int32_t k, void* y, void* workspace, size_t ws_bytes, moe_stream_t stream,
            const moe_debug* debug) {
  return run_layer(cfg, wbuf, x, nullptr, nullptr, nullptr, logits, T, k, y, workspace, ws_bytes,
                   stream, debug);
}

int moe_run_quantized(const moe_config* cfg, const void* wbuf, const uint8_t* xq,
                      const uint8_t* xsf, const float* ts_a, const float* logits, int32_t T,
                      int32_t k, void* y, void* workspace, size_t ws_bytes, moe_stream_t stream,
                      const moe_debug* debug) {
  if (T > 0 && (!xq || !xsf || !ts_a)) return MOE_ERR_INVALID_ARG;
  return run_layer(cfg, wbuf, nullptr, xq, xsf, ts_a, logits, T, k, y, workspace, ws_bytes,
                   stream, debug);
}

int moe_last_device_status(const void* workspace, int32_t* host_status) {
  if (!workspace || !host_status) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(host_status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
