/*
 * nvfp4_moe.h - C ABI of the fused NVFP4 Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * The layer (one call of moe_run):
 *   1. router: softmax over E logits per token, top-k under the strict order (value descending,
 *      lower expert index on ties), weights renormalised over the chosen k
 *      ("vllm.cpp docs/STATUS.md", row "DeepSeek-V4-Flash decode ds4-gap - Lever 3");
 *   2. activation quantiser: x [T,H] BF16 -> NVFP4 with one FP32 tensor scale max|x|/(6*448)
 *      ("nvfp4-megamoe-kernel compare pre-b1...master", section "7. NVFP4 Quantization / Runtime
 *      Activation Global Scale (gsa)"), E4M3 scales per 16 elements, E2M1 codes;
 *   3. plan: per-expert counts, offsets and a stable token->expert permutation, built on the device
 *      without any host read (same page, "CATEGORY 3: Data-dependent control flow" - bincount
 *      replaced by a device scatter into a preallocated buffer - and "SECTION C - DSV4-specific
 *      kernels that must be GPU-native", item 4: expert offsets stay GPU tensors);
 *   4. GEMM1: block-scaled FP4 grouped GEMM of the gathered rows with each expert's gate and up
 *      weights, epilogue SwiGLU silu(g)*u and NVFP4 requantisation of h (same page, section "MoE
 *      kernel (FusedSwiGLUScaledGroupedGemmKernel)");
 *   5. GEMM2: block-scaled FP4 grouped GEMM of h with the down weights, scaled by the router weight;
 *   6. combine: y[t] = sum_j w_j * out_j (+ the shared expert, weight 1), rounded once to BF16
 *      ("vllm.cpp docs/STATUS.md", row "Brick C part 1", MoeCombineKernel).
 *
 * Formats.  NVFP4 codes are E2M1, two per byte, element 2i in the low nibble; block scales are
 * FP8 E4M3 (one byte per 16 consecutive elements along the reduction dimension); tensor scales
 * are FP32.  Canonical layouts are row major: codes [rows, cols/2], scales [rows, cols/16].
 *
 * Conventions for every entry point.
 *   - Tensor pointers are DEVICE pointers unless stated otherwise; tensors are contiguous and row
 *     major; BF16 tensors are passed as void*.
 *   - The caller owns every buffer: inputs, outputs, the packed-weight buffer and the workspace.
 *     The library allocates no memory and keeps no state between calls.
 *   - All work is enqueued on `stream`; no entry point synchronises except
 *     moe_last_device_status.  moe_quantize_act, moe_plan and moe_run read nothing back to the
 *     host and allocate nothing, so they can be recorded in a CUDA graph.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Argument errors are detected on the
 *     host before anything is enqueued.  Errors found on the device (a non-finite activation
 *     maximum, a pipeline wait that ran out) are written to a status word at the start of the
 *     workspace; read it with moe_last_device_status.  Outputs of a call that raised a device
 *     error are unspecified.
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,       /* null pointer, k < 1 or k > E, negative size ... */
  MOE_ERR_UNSUPPORTED_SHAPE = -2, /* H or I not a multiple of 32, T > max_tokens, E > 1024 ... */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3,
  MOE_ERR_CUDA = -4,              /* a CUDA runtime call failed (launch error ...) */
  MOE_ERR_DEVICE_TIMEOUT = -5,    /* device status: a bounded pipeline wait ran out */
  MOE_ERR_NONFINITE = -6,         /* device status: max|x| is not finite */
  MOE_ERR_UNIMPLEMENTED = -7
} moe_status;

/* Shape of one MoE layer. */
typedef struct {
  int32_t num_experts;   /* E, routed experts, 1..1024 */
  int32_t hidden;        /* H, multiple of 32 (16-byte code rows); see the note below */
  int32_t inter;         /* I, routed-expert intermediate size, multiple of 32 */
  int32_t top_k;         /* k, 1..min(E, 32) */
  int32_t shared_inter;  /* 0: no shared expert; otherwise its intermediate size, a multiple of 32
                            (one other than I runs, like an unaligned width, padded: see below) */
  float h_tensor_scale;  /* fixed FP32 tensor scale used to requantise h (1.0 by default) */
  int32_t max_tokens;    /* largest T a workspace sized with moe_workspace_size must serve */
  uint32_t flags;        /* MOE_FLAG_* variant bits below; 0 = the base layer */
  float swiglu_limit;    /* L of MOE_FLAG_SWIGLU_CLAMP and MOE_FLAG_ACT_SWIGLU_OAI: finite, >= 0 */
  float swiglu_alpha;    /* slope of MOE_FLAG_ACT_SWIGLU_OAI (1.702 in gpt-oss): finite */
} moe_config;

/* Widths.  H, I and the shared expert's intermediate size need only be multiples of 32.  A width
 * that is not a multiple of 256 (the K stage of the packed weight blocks), or a shared expert
 * whose intermediate size differs from I, is padded inside the library: H runs rounded up to a
 * multiple of 256, and both intermediate sizes run at the larger of the two rounded up to a
 * multiple of 256.  The weight buffer holds zero rows and columns up to those widths
 * (moe_weights_size counts them), and moe_run / moe_run_quantized copy x (or its codes and
 * scales) into zero-padded rows of the workspace and the output rows back into y
 * (moe_workspace_size counts both buffers).  Debug rows of h are as wide as the larger
 * intermediate size (a narrower expert's rows end in zeros).  The results are those of the
 * unpadded layer: a padded column of x meets only zero weights, and a padded feature of h is
 * activation(0, 0) = 0 for every activation flag, quantised to a zero block. */

/* Router variant ("vllm.cpp docs/STATUS.md", paragraph "W6 sqrtsoftplus + hash-routed MoE";
 * "nvfp4-megamoe-kernel compare pre-b1...master", section "Dense Router (L3+)"): expert scores
 * s_e = sqrt(softplus(logit_e)) (softplus(x) = x above 20), top-k selection on s_e + bias_e (the
 * per-expert correction bias set with moe_set_router_bias; zero by default), weights
 * w_j = s_(e_j) / sum of the k chosen s (in slot order).  Without the flag: top-k of the logits,
 * softmax renormalised over the k. */
#define MOE_FLAG_ROUTER_SQRTSOFTPLUS 1u
/* Activation variant (same paragraph; "nvfp4-megamoe-kernel ...", section "Nvfp4MoE (Routed
 * Experts)", swiglu_limit = 10): h = silu(min(g, L)) * clamp(u, -L, L); L = 0 zeroes every
 * expert.  Without the flag: h = silu(g) * u. */
#define MOE_FLAG_SWIGLU_CLAMP 2u
/* The other two activations of the pages' MoE ("b12x" README, section "What's in here", moe:
 * "with SiLU/ReLU2/SwiGLU-OAI activations"; SiLU is the base SwiGLU).  The pages give only their
 * names; the formulas are the published definitions.  At most one activation flag is set.
 *   MOE_FLAG_ACT_RELU2: non-gated experts, h = max(u, 0)^2 with u the up projection alone.  The
 *     experts have no gate matrix: moe_quantize_weights ignores w_gate / s_gate (pass NULL), GEMM1
 *     has I output rows per expert instead of 2I, and moe_weights_export of matrix 0 is an error.
 *   MOE_FLAG_ACT_SWIGLU_OAI: the gpt-oss SwiGLU, g' = min(g, L), u' = clamp(u, -L, L),
 *     h = (u' + 1) * g' * sigmoid(alpha * g') with L = swiglu_limit, alpha = swiglu_alpha. */
#define MOE_FLAG_ACT_RELU2 4u
#define MOE_FLAG_ACT_SWIGLU_OAI 8u
/* W4A16 activation precision ("b12x" README, section "What's in here", moe: "W4A16 (BF16
 * activations, inline FP4 weight dequant - no activation-scale math)"): the BF16 x enters the
 * gate/up GEMM as it is (no activation quantiser, no tensor scale), the NVFP4 weights are
 * decoded to BF16 inside the GEMMs (BF16 tensor-core MMAs), and h is rounded to BF16 (nearest
 * even) before the down projection; routing, plan and combine are those of the base layer.  Any
 * activation flag may be combined with it.  The weights are the same NVFP4 buffer.  In the
 * debug struct, hq / hsf are not written and hb receives h. */
#define MOE_FLAG_ACT_BF16 16u
/* W4A8 activation precision ("b12x" README, section "DeepSeek V4 Flash 0731 MoE reproduction":
 * "MXFP4 E8M0/K32 weights, MXFP8 activations"): the weights are MXFP4 (E2M1 codes, one E8M0
 * scale 2^(byte - 127) per 32 along K, no tensor scale) instead of NVFP4; x is quantised to
 * MXFP8 (E4M3 codes, one E8M0 scale per 32, no tensor scale) and h is requantised to MXFP8.  The
 * scale byte of a block is 2^(floor(log2 max|v|) - emax), emax = 2 for E2M1 and 8 for E4M3,
 * clamped to [0, 254] (0 for an all-zero block); elements are v / scale rounded to nearest even
 * and saturated.  The GEMMs decode both operands exactly to BF16 and run on the BF16 tensor cores.
 * moe_weights_export returns E8M0 scales [N, K/32] (and ts = 1); in the debug struct xq / xsf
 * receive the MXFP8 codes [T, H] and scales [T, H/32] of x, hq / hsf those of h ([rows, I],
 * [rows, I/32]) and hb its decoded BF16 values.  Not combinable with MOE_FLAG_ACT_BF16. */
#define MOE_FLAG_ACT_MXFP8 32u

/* Optional device buffers that receive the layer's intermediates (any field may be NULL). */
typedef struct {
  int32_t* topk_ids; /* [T,k] */
  float* topk_w;     /* [T,k] */
  int32_t* counts;   /* [E] */
  int32_t* offsets;  /* [E+1] */
  int32_t* perm_src; /* [T*k] permuted row -> token */
  int32_t* inv;      /* [T*k] assignment t*k+j -> permuted row */
  uint8_t* xq;       /* [T,H/2]  quantised activations */
  uint8_t* xsf;      /* [T,H/16] */
  float* ts_a;       /* [1]      activation tensor scale */
  uint8_t* hq;       /* [T*k + T*shared, I/2]  requantised intermediate, permuted row order,
                        shared-expert rows last (row T*k + t is token t) */
  uint8_t* hsf;      /* [T*k + T*shared, I/16] */
  void** stage_events; /* NULL, or an array of MOE_STAGE_EVENTS cudaEvent_t handles recorded on
                          `stream`: [0] before the layer, then after the activation quantiser,
                          the router + plan, GEMM1, GEMM2 and the BF16 output respectively */
  uint32_t inject;     /* test hooks for the failure path, MOE_INJECT_* bits; 0 in normal use */
  void* hb;            /* [T*k + T*shared, I] BF16 h of a MOE_FLAG_ACT_BF16 layer, same row order as
                          hq */
} moe_debug;

#define MOE_STAGE_EVENTS 6
/* Decode-sized batches: the prologue never raises the flag that tells the grouped-GEMM launch
 * its plan is ready, so that launch's bounded wait (about 2 s) runs out before it issues any
 * copy; the call then leaves MOE_ERR_DEVICE_TIMEOUT in the device status and unspecified
 * output, and the next call without the hook runs normally.  It tests the timeout path without
 * faulting or hanging the GPU; the pages have no counterpart. */
#define MOE_INJECT_NO_PLAN_FLAG 1u

/* Text for a status code (static storage). */
const char* moe_status_string(int status);

/* Checks a configuration; MOE_OK or the error moe_run would return for it. */
int moe_config_check(const moe_config* cfg);

/* ---------------------------------------------------------------------------------------------
 * Weights.  moe_quantize_weights turns BF16 expert weights into NVFP4 (per expert and matrix: an
 * FP32 tensor scale max|W|/(6*448), E4M3 block scales along the input dimension, E2M1 codes;
 * "nvfp4-megamoe-kernel compare pre-b1...master", section "NVFP4 Weight Global Scale (gsb)", and
 * "vllm.cpp docs/STATUS.md" row on NVFP4 weight_packed [N, K/2] / weight_scale [N, K/16]) and
 * writes them into a caller-owned device buffer of moe_weights_size bytes, in the library's
 * private GEMM-ready layout (gate/up rows interleaved by 16, scales pre-arranged for the tensor
 * memory copy).  Off the hot path: run once per layer.
 * ------------------------------------------------------------------------------------------- */
size_t moe_weights_size(const moe_config* cfg);

/* w_gate, w_up: [E, I, H] BF16; w_down: [E, H, I] BF16; s_gate, s_up: [I, H], s_down: [H, I]
 * (NULL unless cfg->shared_inter > 0; w_gate and s_gate are not read, and may be NULL, with
 * MOE_FLAG_ACT_RELU2).  wbuf: 256-byte aligned device buffer of wbuf_bytes.
 * Returns MOE_ERR_INVALID_ARG on null pointers, MOE_ERR_WORKSPACE_TOO_SMALL if wbuf_bytes is too
 * small.  Non-finite weights give unspecified codes. */
int moe_quantize_weights(const moe_config* cfg, const void* w_gate, const void* w_up,
                         const void* w_down, const void* s_gate, const void* s_up,
                         const void* s_down, void* wbuf, size_t wbuf_bytes, moe_stream_t stream);

/* Stores the router's per-expert selection bias (bias: device FP32 [E], copied) into wbuf, where
 * MOE_FLAG_ROUTER_SQRTSOFTPLUS layers read it; moe_quantize_weights leaves it zero.  The bias
 * only changes which experts are chosen, never their weights.  MOE_ERR_INVALID_ARG on null
 * pointers. */
int moe_set_router_bias(const moe_config* cfg, void* wbuf, const float* bias, moe_stream_t stream);

/* Copies one expert matrix back out of wbuf in canonical layout.  expert: 0..E-1, or -1 for the
 * shared expert; matrix: 0 gate [I,H], 1 up [I,H], 2 down [H,I].  codes [N, K/2], sf [N, K/16]
 * and ts [1] are device buffers. */
int moe_weights_export(const moe_config* cfg, const void* wbuf, int32_t expert, int32_t matrix,
                       uint8_t* codes, uint8_t* sf, float* ts, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Activation quantiser (one tensor scale for the whole [rows, cols] tensor, then per-16 blocks).
 * x: [rows, cols] BF16, cols a multiple of 16 and x 16-byte aligned; codes [rows, cols/2];
 * sf [rows, cols/16]; ts: device FP32 scalar.  rows == 0 is MOE_OK and does nothing.
 * ------------------------------------------------------------------------------------------- */
size_t moe_act_workspace_size(int64_t rows, int64_t cols);
int moe_quantize_act(const void* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                     float* ts, void* workspace, size_t ws_bytes, moe_stream_t stream);

/* RMSNorm followed by the activation quantiser: the producer that feeds the layer's quantised
 * input ("nvfp4-megamoe-kernel compare pre-b1...master", sections "P4 - Fused RMSNorm + NVFP4
 * quantize" and "P5": two kernels, no BF16 round trip between the norm and the quantiser; its
 * output goes straight into moe_run_quantized).  Per row: ms = (sum of x^2) / cols,
 * r = 1 / sqrt(ms + eps), y = (x * r) * gamma, all FP32; then one tensor scale max|y| / 2688 for
 * the whole tensor and the per-16 encode of y, as moe_quantize_act does for x.  The sum of
 * squares is defined as the exact sum rounded once to FP32; the kernel forms it in FP32 in its
 * own (coalesced) order, within (7 + 5 + log2(ceil(cols / 256))) * 2^-24 of the exact sum
 * relative, so r, ts and the few codes whose quotients lie that close to a rounding boundary may
 * differ from the exact definition by one step.  x: [rows, cols] BF16, gamma: [cols] BF16, both
 * 16-byte aligned, cols a multiple of 16 and at most 16384; codes [rows, cols/2],
 * sf [rows, cols/16], ts: device FP32 scalar; rrms: NULL or device FP32 [rows] that receives
 * each row's r.  workspace: >= moe_rmsnorm_workspace_size(rows) bytes (its first word is the
 * device status: MOE_ERR_NONFINITE when max|y| is not finite).  rows == 0 is MOE_OK. */
size_t moe_rmsnorm_workspace_size(int64_t rows);
int moe_rmsnorm_quantize_act(const void* x, const void* gamma, float eps, int64_t rows,
                             int64_t cols, uint8_t* codes, uint8_t* sf, float* ts, float* rrms,
                             void* workspace, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Router + plan.  logits [T,E] FP32 -> topk_ids [T,k] (slot 0 the largest), topk_w [T,k],
 * counts [E], offsets [E+1] (exclusive prefix sums, offsets[E] = T*k), perm_src [T*k]
 * (permuted row -> token; rows of one expert ordered by ascending t*k+j), inv [T*k].
 * ------------------------------------------------------------------------------------------- */
size_t moe_plan_workspace_size(int32_t T, int32_t E, int32_t k);
int moe_plan(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
             float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv,
             void* workspace, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_plan_static: moe_plan without a workspace argument.  It has no counterpart on the pages
 * this library follows; it exists for callers that cannot allocate device memory (a plugin whose
 * host framework owns every device allocation, code running while a memory pool is frozen or
 * capped, a plain C caller without an allocator).  Its scratch is a file-scope static device
 * array of MOE_PLAN_STATIC_SCRATCH_BYTES bytes that every GPU loading the library keeps until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Arguments and outputs are those of moe_plan; the caller still owns every output buffer.
 *   - A problem whose moe_plan_workspace_size(T, E, k) exceeds MOE_PLAN_STATIC_SCRATCH_BYTES is
 *     rejected with MOE_ERR_WORKSPACE_TOO_SMALL: ceil(T/64)*E (ceil(T/32)*E for k > 16) must
 *     stay within about 130,000, e.g. up to T = 8,128 tokens at E = 1,024 experts, 32,704 at
 *     E = 256, 65,472 at E = 128.
 *   - Every call that is not being recorded into a CUDA graph looks up the array's device
 *     address (cudaGetSymbolAddress) on the current device, so a device reset, which may move
 *     the array, is picked up by the next call.  A call made during stream capture reuses the
 *     address found by the last uncaptured call on that device: make the first call on a device,
 *     and the first call after a reset, outside any capture (a captured call with no earlier
 *     lookup returns MOE_ERR_CUDA).
 *   - All calls share the one array per device, and it keeps the last call's contents: calls
 *     that may overlap on the GPU (two streams, two threads) race and must be serialised by the
 *     caller.  The device status word in the array is cleared at the start of every call.
 * ------------------------------------------------------------------------------------------- */
#define MOE_PLAN_STATIC_SCRATCH_BYTES (1u << 20)
int moe_plan_static(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
                    float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm_src,
                    int32_t* inv, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * The layer.  wbuf: written by moe_quantize_weights for the same cfg.  x [T,H] BF16 (16-byte
 * aligned), logits [T,E] FP32, y [T,H] BF16 out.  k must equal cfg->top_k.  T == 0 is MOE_OK.
 * workspace: >= moe_workspace_size(cfg, T) bytes, 256-byte aligned.  debug: NULL, or a host
 * struct of device buffers that receive the intermediates.
 * ------------------------------------------------------------------------------------------- */
size_t moe_workspace_size(const moe_config* cfg, int32_t T);

/* Number of kernels one moe_run(cfg, ..., T, ...) launches (memset nodes not counted), or a
 * negative moe_status for an invalid cfg / T.  Host-only arithmetic: no CUDA call, no device.
 * It mirrors moe_run's choice of path: 3 for decode-sized batches (cluster prologue, both grouped
 * GEMMs in one persistent launch, row sum), 5 for other small batches, 6 or 8 for large ones (the router and plan take one
 * kernel up to 2048 routed rows, three above).  A utility for launch accounting; the pages have
 * no counterpart. */
int moe_run_kernel_count(const moe_config* cfg, int32_t T);
int moe_run(const moe_config* cfg, const void* wbuf, const void* x, const float* logits, int32_t T,
            int32_t k, void* y, void* workspace, size_t ws_bytes, moe_stream_t stream,
            const moe_debug* debug);

/* The layer on activations that are already NVFP4 (the output of moe_quantize_act or of the
 * fused RMSNorm producer moe_rmsnorm_quantize_act): the router, plan, both grouped GEMMs and the
 * combine of moe_run, without the BF16 read and the activation quantiser, so the normalised
 * activations never make a BF16 round trip ("nvfp4-megamoe-kernel compare pre-b1...master",
 * sections "P4 - Fused RMSNorm + NVFP4 quantize" and "P5": the norm's quantised output feeds the
 * MoE directly).  xq [T, H/2] E2M1 codes (16-byte aligned), xsf [T, H/16] E4M3 scales (4-byte
 * aligned) and ts_a (device FP32 scalar, the tensor scale the codes were made with) are read
 * as they are; everything else as for moe_run, with the same workspace size, launch count and
 * output.  A negative, NaN or infinite *ts_a sets MOE_ERR_NONFINITE in the device status. */
int moe_run_quantized(const moe_config* cfg, const void* wbuf, const uint8_t* xq,
                      const uint8_t* xsf, const float* ts_a, const float* logits, int32_t T,
                      int32_t k, void* y, void* workspace, size_t ws_bytes, moe_stream_t stream,
                      const moe_debug* debug);

/* Synchronises `stream`'s device and copies the device status word at the start of a workspace
 * used by moe_quantize_act, moe_plan or moe_run into *host_status (MOE_OK or a device error). */
int moe_last_device_status(const void* workspace, int32_t* host_status);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_MOE_H */
