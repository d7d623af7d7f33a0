// NVFP4 Mixture-of-Experts layer: plain, slow, single-threaded CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load or call this file: only the
// tests, the smoke check and the CPU-baseline leg of the benchmark use it.  It shares no code,
// table or header with the CUDA library; it is written from the format and layer definitions.
// Build with -ffp-contract=off so that every FP32 product and sum is rounded on its own (the
// sequential-FP32 arithmetic below is the definition, on x86-64 and on AArch64 alike).
// The same source builds a second time with -fopenmp for the all-core CPU baseline: the only
// parallel loops run over independent experts, rows or tokens (each writes its own outputs with
// its own scratch), and every sum inside a row keeps its sequential order, so both builds give
// identical bits.  The maxima use max, which is exact in any order.
//
// Definitions followed (page title, section):
//  * NVFP4 = E2M1 values, FP8 E4M3 block scales over 16-element microblocks, FP32 tensor scale:
//    "nvfp4-megamoe-kernel compare pre-b1...master", section "NVFP4 throughout" (weights and
//    activations float4_e2m1fn_x2, scales float8_e4m3fn, MMA kind mxf4nvf4).
//  * Tensor scale = max|X| / (6 * 448): same page, section "7. NVFP4 Quantization / Runtime
//    Activation Global Scale (gsa)"; per-expert weight scale: "NVFP4 Weight Global Scale (gsb)".
//  * Block scale = E4M3(block_amax / 6 / tensor_scale), codes = E2M1(x / (scale * tensor_scale))
//    rounded to nearest even: the layer's problem statement (configuration "Tiny MoE").
//  * Router: softmax, top-k under the strict order (value, lower index on ties), weights
//    renormalised over the k chosen in slot order: "vllm.cpp docs/STATUS.md", row "DeepSeek-V4-
//    Flash decode ds4-gap - Lever 3 (route -> warp-topk)".
//  * Router variant: score sqrt(softplus(logit)), a per-expert correction bias added for the
//    selection only, the weights gathered from the unbiased scores: "vllm.cpp docs/STATUS.md",
//    paragraph "W6 sqrtsoftplus + hash-routed MoE"; "nvfp4-megamoe-kernel ...", section "Dense
//    Router (L3+)" (sqrt(softplus(X @ W_gate)) + e_bias, top-k selection).
//  * Clamped SwiGLU silu(min(g, L)) * clamp(u, -L, L): "vllm.cpp docs/STATUS.md" (gate clamped
//    max-only, up clamped both-sided; a limit of 0 zeroes the expert); L = 10 in "nvfp4-megamoe-
//    kernel ...", section "Nvfp4MoE (Routed Experts)" (swiglu_limit=10.0).
//  * The other activations of the pages' MoE ("b12x" README, section "What's in here", moe:
//    "with SiLU/ReLU2/SwiGLU-OAI activations"): ReLU2 is the squared ReLU of a non-gated expert,
//    h = max(u, 0)^2 with u the up projection alone (no gate matrix); SwiGLU-OAI is the clamped
//    variant h = (clamp(u, -L, L) + 1) * g' * sigmoid(alpha * g'), g' = min(g, L).  The pages give
//    only the names; the formulas are the published definitions of these activations (squared
//    ReLU; the gpt-oss SwiGLU with its alpha = 1.702 and limit 7 as the defaults of the tests).
//  * SwiGLU silu(g)*u on FP32 accumulators in the GEMM1 epilogue: "nvfp4-megamoe-kernel ...",
//    section "MoE kernel (FusedSwiGLUScaledGroupedGemmKernel)"; shared expert with weight 1:
//    section "6. MoE (Mixture of Experts) / Nvfp4SharedExpert".
//  * Weighted combine y = sum_j w_j * expert_out_j: "vllm.cpp docs/STATUS.md", row "Brick C part 1"
//    (MoeCombineKernel).
//  * W4A16 activation precision: BF16 activations enter the expert GEMMs as they are (no
//    activation scale), the NVFP4 weights are decoded at the point of use: "b12x" README,
//    section "What's in here" (moe: "W4A16 (BF16 activations, inline FP4 weight dequant - no
//    activation-scale math)").
//  * W4A8 activation precision: MXFP4 weights (E2M1 values, one E8M0 scale per 32 elements along
//    K) and MXFP8 activations (E4M3 values, one E8M0 scale per 32), no tensor scale: "b12x"
//    README, section "DeepSeek V4 Flash 0731 MoE reproduction" ("MXFP4 E8M0/K32 weights, MXFP8
//    activations"); E8M0 = 2^(byte - 127), group 32, no global scale: "vllm.cpp docs/STATUS.md",
//    the MXFP4 weight-dequant row; "four E8M0 scales, one per 32 values": "b12x" README (the
//    compressed all-reduce modes).
//
// Readings where the pages are silent (each also listed in the design notes):
//  * two E2M1 codes per byte, element 2i in the low nibble;
//  * a negative value that rounds to zero keeps its sign (code 0x8);
//  * E4M3 encoding rounds to nearest even and saturates finite overflow (and +inf) to 448;
//  * a block whose max |x| is 0, or whose decoded scale is 0, gets scale byte 0 and all codes 0;
//  * one activation tensor scale for the whole [T, H] input;
//  * the intermediate h is requantised with a fixed tensor scale (default 1.0);
//  * rows of one expert are ordered by ascending flat assignment index t*k + j (stable);
//  * no rounding between stages: g, u, h, the down projection and the combine stay FP32 and the
//    output is rounded once to BF16 (nearest even);
//  * softplus(x) = x for x > 20, log1p(exp(x)) otherwise (FP32); the variant router's weights are
//    the chosen unbiased scores divided by their sum (summed in slot order), as the base router
//    renormalises over the k chosen;
//  * W4A16: the intermediate h is rounded to BF16 (nearest even) before the down projection, the
//    16-bit activation format of that path; everything else is the base layer;
//  * MX block scale (the pages give only the decode rule): 2^(floor(log2 max|x|) - emax) with emax
//    the exponent of the element format's largest power of two (E4M3: 8, E2M1: 2), the byte
//    clamped to [0, 254], byte 0 for an all-zero block; elements x / scale rounded to nearest even
//    and saturated (to 448 or 6); W4A8 requantises h to MXFP8 the same way.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// Thread count of the OpenMP build (n <= 0: all host cores); the single-threaded build ignores it.
void orc_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
  (void)n;
#endif
}

int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// ---------------------------------------------------------------------------------------------
// Scalar formats
// ---------------------------------------------------------------------------------------------

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round-to-nearest-even FP32 -> BF16 (NaN stays a quiet NaN).
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

// E2M1: sign bit 3; magnitude by the 3-bit code, exponent bias 1, one mantissa bit:
//   000 0, 001 0.5 (subnormal), 010 1, 011 1.5, 100 2, 101 3, 110 4, 111 6.
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_e2m1_decode(uint8_t c) {
  float m = kE2M1[c & 7];
  return (c & 8) ? -m : m;
}

// Nearest E2M1 value to q, ties to the even code (= even mantissa bit); |q| > 6 saturates to 6.
uint8_t orc_e2m1_encode(float q) {
  float a = std::fabs(q);
  uint8_t m;
  if (a <= 0.25f) m = 0;       // tie 0.25 -> 0 (even)
  else if (a < 0.75f) m = 1;   // tie 0.75 -> 1.0 (code 2, even)
  else if (a <= 1.25f) m = 2;  // tie 1.25 -> 1.0
  else if (a < 1.75f) m = 3;   // tie 1.75 -> 2.0
  else if (a <= 2.5f) m = 4;   // tie 2.5 -> 2.0
  else if (a < 3.5f) m = 5;    // tie 3.5 -> 4.0
  else if (a <= 5.0f) m = 6;   // tie 5 -> 4.0
  else m = 7;
  return (uint8_t)(m | (std::signbit(q) ? 8 : 0));
}

// E4M3 ("fn" variant): bias 7, exponent field 0 subnormal m/8 * 2^-6, 0x7F/0xFF NaN, no inf.
float orc_e4m3_decode(uint8_t c) {
  int e = (c >> 3) & 15, m = c & 7;
  float v;
  if (e == 15 && m == 7) v = NAN;
  else if (e == 0) v = std::ldexp((float)m, -9);
  else v = std::ldexp((float)(8 + m), e - 10);
  return (c & 0x80) ? -v : v;
}

// Nearest E4M3 value, ties to even mantissa; finite overflow and inf saturate to +-448.
uint8_t orc_e4m3_encode(float v) {
  if (std::isnan(v)) return 0x7F;
  uint8_t s = std::signbit(v) ? 0x80 : 0x00;
  float a = std::fabs(v);
  if (a >= 448.0f) return s | 0x7E;
  if (a == 0.0f) return s;
  int ex;
  std::frexp(a, &ex);  // a = f * 2^ex with f in [0.5, 1)
  int E = ex - 1;      // floor(log2 a)
  if (E < -6) {        // subnormal range: spacing 2^-9
    int m = (int)std::nearbyint(std::ldexp(a, 9));
    if (m == 8) return s | 0x08;  // rounded up to the smallest normal 2^-6
    return (uint8_t)(s | m);
  }
  int m8 = (int)std::nearbyint(std::ldexp(a, 3 - E));  // in [8, 16]
  if (m8 == 16) { E += 1; m8 = 8; }
  int code = ((E + 7) << 3) | (m8 - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(s | code);
}

// ---------------------------------------------------------------------------------------------
// NVFP4 quantisation
// ---------------------------------------------------------------------------------------------

// One 16-element block with tensor scale ts: writes 8 code bytes and 1 scale byte.
static void quant_block16(const float* x, float ts, uint8_t* codes8, uint8_t* sf) {
  float bamax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = std::fabs(x[i]);
    if (a > bamax) bamax = a;
  }
  if (bamax == 0.0f) {
    *sf = 0;
    std::memset(codes8, 0, 8);
    return;
  }
  float t = bamax / 6.0f;
  t = t / ts;
  uint8_t s = orc_e4m3_encode(t);
  *sf = s;
  float S = orc_e4m3_decode(s) * ts;
  if (S == 0.0f) {
    std::memset(codes8, 0, 8);
    return;
  }
  for (int i = 0; i < 8; ++i) {
    uint8_t lo = orc_e2m1_encode(x[2 * i] / S);
    uint8_t hi = orc_e2m1_encode(x[2 * i + 1] / S);
    codes8[i] = (uint8_t)(lo | (hi << 4));
  }
}

// Quantise FP32 rows [rows, cols] (cols % 16 == 0) with a given tensor scale.
void orc_quantize_f32(const float* x, int64_t rows, int64_t cols, float ts, uint8_t* codes,
                      uint8_t* sf) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < cols / 16; ++b)
      quant_block16(x + r * cols + b * 16, ts, codes + r * (cols / 2) + b * 8,
                    sf + r * (cols / 16) + b);
}

// Tensor scale of a BF16 tensor: max|x| / 2688 (2688 = 6 * 448, exact in FP32).
float orc_tensor_scale_bf16(const uint16_t* x, int64_t n) {
  float amax = 0.0f;
  int nan = 0;
#pragma omp parallel for reduction(max : amax) reduction(| : nan)
  for (int64_t i = 0; i < n; ++i) {
    float a = std::fabs(orc_bf16_to_f32(x[i]));
    if (std::isnan(a)) nan = 1;
    else if (a > amax) amax = a;
  }
  if (nan) return NAN;
  return amax / 2688.0f;
}

// Full NVFP4 quantisation of a BF16 tensor [rows, cols]: tensor scale, block scales, codes.
// Returns 0, or -6 when the tensor holds a non-finite value.
int orc_quantize_bf16(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                      float* ts_out) {
  float ts = orc_tensor_scale_bf16(x, rows * cols);
  *ts_out = ts;
  if (!std::isfinite(ts)) return -6;
#pragma omp parallel
  {
    std::vector<float> row(cols);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      for (int64_t c = 0; c < cols; ++c) row[c] = orc_bf16_to_f32(x[r * cols + c]);
      orc_quantize_f32(row.data(), 1, cols, ts, codes + r * (cols / 2), sf + r * (cols / 16));
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------------------------
// MX formats (W4A8): one E8M0 scale per 32 elements, no tensor scale
// ---------------------------------------------------------------------------------------------

// E8M0: the byte is a biased exponent, value 2^(b - 127); 0xFF is NaN.
float orc_e8m0_decode(uint8_t b) {
  if (b == 0xFF) return NAN;
  return std::ldexp(1.0f, (int)b - 127);
}

// Scale byte of a block with max |x| = amax for elements whose largest power of two is 2^emax:
// 2^(floor(log2 amax) - emax), the byte clamped to [0, 254]; amax = 0 gives byte 0.
uint8_t orc_mx_scale(float amax, int emax) {
  if (!(amax > 0.0f)) return 0;
  int e = 0;
  std::frexp(amax, &e);  // amax = m * 2^e, m in [0.5, 1): floor(log2 amax) = e - 1
  int b = (e - 1) - emax + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return (uint8_t)b;
}

// kind 0: MXFP8 (E4M3 elements, one byte each); kind 1: MXFP4 (E2M1, two per byte, element 2i in
// the low nibble).  Rows [rows, cols], cols % 32 == 0; scales [rows, cols / 32].
void orc_mx_quantize_f32(const float* x, int64_t rows, int64_t cols, int kind, uint8_t* codes,
                         uint8_t* scales) {
  const int emax = kind == 0 ? 8 : 2;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < cols / 32; ++b) {
      const float* xb = x + r * cols + b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(xb[i]));
      const uint8_t sb = orc_mx_scale(amax, emax);
      scales[r * (cols / 32) + b] = sb;
      const float X = orc_e8m0_decode(sb);
      for (int i = 0; i < 32; ++i) {
        const float q = xb[i] / X;
        const int64_t c = r * cols + b * 32 + i;
        if (kind == 0) {
          codes[c] = orc_e4m3_encode(q);
        } else {
          const uint8_t nib = orc_e2m1_encode(q);
          uint8_t& byte = codes[c / 2];
          byte = (c & 1) ? (uint8_t)((byte & 0x0F) | (nib << 4)) : (uint8_t)((byte & 0xF0) | nib);
        }
      }
    }
}

// v = element * 2^(scale byte - 127).
void orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                       int kind, float* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const int64_t i = r * cols + c;
      float v;
      if (kind == 0) {
        v = orc_e4m3_decode(codes[i]);
      } else {
        const uint8_t byte = codes[i / 2];
        v = orc_e2m1_decode((i & 1) ? (byte >> 4) : (byte & 15));
      }
      out[i] = v * orc_e8m0_decode(scales[r * (cols / 32) + c / 32]);
    }
}

// v = (e2m1(code) * e4m3(sf)) * ts, rows [rows, cols].
// RMSNorm then NVFP4 quantisation of x [rows, cols] BF16 with gamma [cols] BF16 (the producer
// feeding the layer's activation quantiser: "nvfp4-megamoe-kernel compare pre-b1...master",
// sections "P4 - Fused RMSNorm + NVFP4 quantize" and "P5"; two passes, the tensor scale taken
// from the normalised values).  The pages leave the summation order of the mean square open; the
// reading taken is the plain one: the sum of the squares, accumulated in float64 (each square of
// a BF16 value is exact in float64, and the float64 sum of up to 2^14 of them is within
// n * 2^-53 of the exact sum, far below the FP32 rounding that follows) and rounded once to FP32.
// Then ms = sum / cols, r = 1 / sqrt(ms + eps), y_c = (x_c * r) * gamma_c (FP32, in that order);
// ts = max|y| / 2688 over the whole tensor and the block encode of y (as orc_quantize_f32).
// Writes y [rows, cols] if y_out is not null and each row's r into r_out if it is not null.
// Returns -6 when max|y| is not finite.
float orc_sum_squares(const float* v, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += (double)v[i] * (double)v[i];
  return (float)s;
}

int orc_rmsnorm_quantize(const uint16_t* x, const uint16_t* gamma, float eps, int64_t rows,
                         int64_t cols, uint8_t* codes, uint8_t* sf, float* ts_out, float* y_out,
                         float* r_out) {
  std::vector<float> y((size_t)rows * cols), row(cols);
  float amax = 0.0f;
  bool nan = false;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; ++c) row[c] = orc_bf16_to_f32(x[r * cols + c]);
    const float ms = orc_sum_squares(row.data(), cols) / (float)cols;
    const float rinv = 1.0f / std::sqrt(ms + eps);
    if (r_out) r_out[r] = rinv;
    for (int64_t c = 0; c < cols; ++c) {
      const float v = (row[c] * rinv) * orc_bf16_to_f32(gamma[c]);
      y[r * cols + c] = v;
      const float a = std::fabs(v);
      if (std::isnan(a)) nan = true;
      else if (a > amax) amax = a;
    }
  }
  const float ts = nan ? NAN : amax / 2688.0f;
  *ts_out = ts;
  if (y_out) std::copy(y.begin(), y.end(), y_out);
  if (!std::isfinite(ts)) return -6;
  orc_quantize_f32(y.data(), rows, cols, ts, codes, sf);
  return 0;
}

void orc_dequantize(const uint8_t* codes, const uint8_t* sf, float ts, int64_t rows, int64_t cols,
                    float* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = codes[r * (cols / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      float s = orc_e4m3_decode(sf[r * (cols / 16) + c / 16]);
      out[r * cols + c] = (orc_e2m1_decode(code) * s) * ts;
    }
}

// ---------------------------------------------------------------------------------------------
// Router and permutation
// ---------------------------------------------------------------------------------------------

// Per token: k repeated arg-maxes of the raw logits under (value descending, index ascending);
// w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0), summed in slot order (softmax then renormalise
// over the chosen k; softmax is monotone, so selecting on logits selects the same experts).
void orc_router(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w);

float orc_sqrt_softplus(float x) {
  const float sp = x > 20.0f ? x : std::log1p(std::exp(x));
  return std::sqrt(sp);
}

// mode 0: orc_router.  mode 1: per token, s_e = sqrt(softplus(l_e)); k repeated arg-maxes of
// s_e + bias_e (bias may be null: 0) under (value descending, index ascending); w_j = s_(e_j) /
// sum_{i<k} s_(e_i), the sum in slot order.
void orc_router_ex(const float* logits, int64_t T, int E, int k, int mode, const float* bias,
                   int32_t* ids, float* w) {
  if (mode == 0) {
    orc_router(logits, T, E, k, ids, w);
    return;
  }
  std::vector<char> taken(E);
  std::vector<float> sc(E), sel(E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    for (int e = 0; e < E; ++e) {
      sc[e] = orc_sqrt_softplus(l[e]);
      sel[e] = sc[e] + (bias ? bias[e] : 0.0f);
    }
    std::fill(taken.begin(), taken.end(), 0);
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || sel[e] > sel[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = best;
      sum = sum + sc[best];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = sc[ids[t * k + j]] / sum;
  }
}

void orc_router(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w) {
  std::vector<char> taken(E);
  std::vector<float> ex(k);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::fill(taken.begin(), taken.end(), 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    float l0 = l[ids[t * k]];
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      ex[j] = std::exp(l[ids[t * k + j]] - l0);
      sum = sum + ex[j];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = ex[j] / sum;
  }
}

// Stable counting sort of the T*k assignments by expert.
void orc_plan(const int32_t* ids, int64_t T, int E, int k, int32_t* counts, int32_t* offsets,
              int32_t* perm_src, int32_t* inv) {
  int64_t R = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < R; ++a) counts[ids[a]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (int64_t a = 0; a < R; ++a) {
    int32_t p = cursor[ids[a]]++;
    perm_src[p] = (int32_t)(a / k);
    inv[a] = p;
  }
}

// ---------------------------------------------------------------------------------------------
// Experts and the layer
// ---------------------------------------------------------------------------------------------

// One expert's quantised weights in canonical layout: gate [I,H], up [I,H], down [H,I]
// (codes [rows, K/2], scales [rows, K/16], K = the input dimension), with their tensor scales.
typedef struct {
  const uint8_t* codes[3];
  const uint8_t* sf[3];
  float ts[3];
} orc_expert;

typedef struct {
  int64_t T;
  int32_t H, I, E, k;
  int32_t has_shared;  // 1: experts[E] is the always-on shared expert (intermediate I_shared)
  int32_t I_shared;
  float ts_h;          // fixed tensor scale of the requantised intermediate
  const uint8_t* xq;   // [T, H/2]   quantised activations
  const uint8_t* xsf;  // [T, H/16]
  float ts_a;
  const float* logits;        // [T, E]
  const orc_expert* experts;  // E + has_shared entries; unreferenced ones may be null
  uint16_t* y;                // [T, H] BF16 out
  // optional outputs (null to skip)
  int32_t* ids;       // [T, k]
  float* w;           // [T, k]
  int32_t* counts;    // [E]
  int32_t* offsets;   // [E + 1]
  int32_t* perm_src;  // [T*k]
  int32_t* inv;       // [T*k]
  uint8_t* hq;        // [T*k, I/2]  routed rows in permuted order
  uint8_t* hsf;       // [T*k, I/16]
  uint8_t* shq;       // [T, I_shared/2]  shared-expert rows
  uint8_t* shsf;      // [T, I_shared/16]
  // variants (zero: the base layer)
  int32_t router_mode;       // 0 softmax over logits, 1 sqrt(softplus) scores + selection bias
  const float* router_bias;  // [E] or null (mode 1 only)
  int32_t swiglu_clamp;      // 1: silu(min(g, L)) * clamp(u, -L, L)
  float swiglu_limit;        // L
  // activation precision (zero: NVFP4 activations, h requantised to NVFP4)
  int32_t act_mode;          // 1: W4A16 - x_bf16 enters GEMM1 as is, h is rounded to BF16;
                             // 2: W4A8 - x_bf16 quantised to MXFP8, experts in MXFP4 (codes
                             //    [N, K/2], sf = E8M0 [N, K/32], ts unused), h requantised to
                             //    MXFP8 (hq / shq [rows, I] E4M3, hsf / shsf [rows, I/32] E8M0)
  const uint16_t* x_bf16;    // [T, H] (act_mode 1 and 2; xq / xsf / ts_a unused)
  uint16_t* hb;              // [T*k, I] BF16 h of the routed rows, permuted order (act_mode 1)
  uint16_t* shb;             // [T, I_shared] BF16 h of the shared expert (act_mode 1)
  float* hf;                 // [T*k, I] FP32 h before its rounding or requantisation (any mode)
  // activation function (zero: SwiGLU, clamped when swiglu_clamp is set)
  int32_t act_kind;          // 1: ReLU2, non-gated: h = max(u, 0)^2 (the gate matrix is unused
                             //    and may be null); 2: SwiGLU-OAI with limit swiglu_limit and
                             //    slope swiglu_alpha
  float swiglu_alpha;
} orc_moe_args;

// h = silu(g) * u, with the optional clamp of gate (from above) and up (both sides) first.
static inline float swiglu(float g, float u, int clamp, float L) {
  if (clamp) {
    g = std::min(g, L);
    u = std::min(std::max(u, -L), L);
  }
  return (g / (1.0f + std::exp(-g))) * u;
}

float orc_swiglu(float g, float u, int clamp, float L) { return swiglu(g, u, clamp, L); }

// Squared ReLU of the up projection (non-gated expert).
static inline float relu2(float u) { return u > 0.0f ? u * u : 0.0f; }

// SwiGLU-OAI: g' = min(g, L), u' = clamp(u, -L, L), h = (u' + 1) * (g' * sigmoid(alpha * g')),
// sigmoid(z) = 1 / (1 + exp(-z)), FP32 in that order.
static inline float swiglu_oai(float g, float u, float L, float alpha) {
  g = std::min(g, L);
  u = std::min(std::max(u, -L), L);
  const float sig = 1.0f / (1.0f + std::exp(-(alpha * g)));
  return (u + 1.0f) * (g * sig);
}

// The activation of one feature from its gate and up values (g unused for ReLU2).
static inline float activation(float g, float u, const orc_moe_args* a) {
  if (a->act_kind == 1) return relu2(u);
  if (a->act_kind == 2) return swiglu_oai(g, u, a->swiglu_limit, a->swiglu_alpha);
  return swiglu(g, u, a->swiglu_clamp, a->swiglu_limit);
}

float orc_activation(float g, float u, int kind, int clamp, float L, float alpha) {
  orc_moe_args a{};
  a.act_kind = kind;
  a.swiglu_clamp = clamp;
  a.swiglu_limit = L;
  a.swiglu_alpha = alpha;
  return activation(g, u, &a);
}

// GEMM1 + SwiGLU, then h requantised to NVFP4 (act_mode 0: codes and scales to hq_row /
// hsf_row) or rounded to BF16 (act_mode 1: bits to hb_row), + GEMM2 for one row: x [H] -> d [H].
static void expert_row(const float* xr, const float* Wg, const float* Wu, const float* Wd, int H,
                       int I, float ts_h, const orc_moe_args* act, int act_mode, float* h,
                       float* hhat, uint8_t* hq_row, uint8_t* hsf_row, uint16_t* hb_row,
                       float* d) {
  for (int n = 0; n < I; ++n) {
    const float* wu = Wu + (int64_t)n * H;
    float g = 0.0f, u = 0.0f;
    if (act->act_kind != 1) {   // ReLU2 experts have no gate
      const float* wg = Wg + (int64_t)n * H;
      for (int c = 0; c < H; ++c) g = g + xr[c] * wg[c];
    }
    for (int c = 0; c < H; ++c) u = u + xr[c] * wu[c];
    h[n] = activation(g, u, act);
  }
  if (act_mode == 1) {
    for (int n = 0; n < I; ++n) {
      hb_row[n] = orc_f32_to_bf16(h[n]);
      hhat[n] = orc_bf16_to_f32(hb_row[n]);
    }
  } else if (act_mode == 2) {
    orc_mx_quantize_f32(h, 1, I, 0, hq_row, hsf_row);
    orc_mx_dequantize(hq_row, hsf_row, 1, I, 0, hhat);
  } else {
    orc_quantize_f32(h, 1, I, ts_h, hq_row, hsf_row);
    orc_dequantize(hq_row, hsf_row, ts_h, 1, I, hhat);
  }
  for (int m = 0; m < H; ++m) {
    const float* wd = Wd + (int64_t)m * I;
    float acc = 0.0f;
    for (int n = 0; n < I; ++n) acc = acc + hhat[n] * wd[n];
    d[m] = acc;
  }
}

static void dequant_expert(const orc_expert& ex, int H, int I, int act_mode,
                           std::vector<float>& Wg, std::vector<float>& Wu, std::vector<float>& Wd) {
  const bool gated = ex.codes[0] != nullptr;   // a ReLU2 expert has no gate matrix
  Wg.resize(gated ? (size_t)I * H : 0);
  Wu.resize((size_t)I * H);
  Wd.resize((size_t)H * I);
  if (act_mode == 2) {  // MXFP4 weights
    if (gated) orc_mx_dequantize(ex.codes[0], ex.sf[0], I, H, 1, Wg.data());
    orc_mx_dequantize(ex.codes[1], ex.sf[1], I, H, 1, Wu.data());
    orc_mx_dequantize(ex.codes[2], ex.sf[2], H, I, 1, Wd.data());
    return;
  }
  if (gated) orc_dequantize(ex.codes[0], ex.sf[0], ex.ts[0], I, H, Wg.data());
  orc_dequantize(ex.codes[1], ex.sf[1], ex.ts[1], I, H, Wu.data());
  orc_dequantize(ex.codes[2], ex.sf[2], ex.ts[2], H, I, Wd.data());
}

// The layer, computed expert by expert over the permuted rows (the oracle proper).
int orc_moe_forward(const orc_moe_args* a) {
  const int64_t T = a->T;
  const int H = a->H, I = a->I, E = a->E, k = a->k;
  const int64_t R = T * k;
  if (T == 0) return 0;
  std::vector<int32_t> ids(R), counts(E), offsets(E + 1), perm_src(R), inv(R);
  std::vector<float> w(R);
  orc_router_ex(a->logits, T, E, k, a->router_mode, a->router_bias, ids.data(), w.data());
  orc_plan(ids.data(), T, E, k, counts.data(), offsets.data(), perm_src.data(), inv.data());

  // the activations entering GEMM1: decoded NVFP4 (act_mode 0), the BF16 values (act_mode 1)
  // or the BF16 values quantised to MXFP8 and decoded (act_mode 2)
  std::vector<float> xhat((size_t)T * H);
  if (a->act_mode == 1 || a->act_mode == 2) {
    for (int64_t i = 0; i < T * H; ++i) xhat[i] = orc_bf16_to_f32(a->x_bf16[i]);
    if (a->act_mode == 2) {
      std::vector<uint8_t> c8((size_t)T * H), s8((size_t)T * H / 32);
      orc_mx_quantize_f32(xhat.data(), T, H, 0, c8.data(), s8.data());
      orc_mx_dequantize(c8.data(), s8.data(), T, H, 0, xhat.data());
    }
  } else {
    orc_dequantize(a->xq, a->xsf, a->ts_a, T, H, xhat.data());
  }

  std::vector<float> D((size_t)R * H);
  const int Imax = std::max(I, a->I_shared);
  const int mx = a->act_mode == 2;
  const int64_t hq_w = mx ? I : I / 2, hs_w = mx ? I / 32 : I / 16;   // bytes per routed h row
  // experts are independent: each writes only its own permuted rows of D, hq, hsf, hb, hf
#pragma omp parallel
  {
    std::vector<float> Wg, Wu, Wd, h(Imax), hhat(Imax);
    std::vector<uint8_t> hq_row(Imax), hsf_row(Imax / 16);   // room for every mode's codes
    std::vector<uint16_t> hb_row(Imax);
#pragma omp for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
      if (counts[e] == 0) continue;
      dequant_expert(a->experts[e], H, I, a->act_mode, Wg, Wu, Wd);
      for (int32_t p = offsets[e]; p < offsets[e + 1]; ++p) {
        const float* xr = xhat.data() + (int64_t)perm_src[p] * H;
        expert_row(xr, Wg.data(), Wu.data(), Wd.data(), H, I, a->ts_h, a, a->act_mode,
                   h.data(), hhat.data(), hq_row.data(), hsf_row.data(), hb_row.data(),
                   D.data() + (int64_t)p * H);
        if (a->act_mode != 1 && a->hq) std::memcpy(a->hq + (int64_t)p * hq_w, hq_row.data(), hq_w);
        if (a->act_mode != 1 && a->hsf) std::memcpy(a->hsf + (int64_t)p * hs_w, hsf_row.data(), hs_w);
        if (a->act_mode == 1 && a->hb) std::copy(hb_row.begin(), hb_row.begin() + I, a->hb + (int64_t)p * I);
        if (a->hf) std::copy(h.begin(), h.begin() + I, a->hf + (int64_t)p * I);
      }
    }
  }
  std::vector<float> S;
  if (a->has_shared) {
    const int Is = a->I_shared;
    S.resize((size_t)T * H);
    std::vector<float> Wg, Wu, Wd;
    dequant_expert(a->experts[E], H, Is, a->act_mode, Wg, Wu, Wd);
    const int64_t shq_w = mx ? Is : Is / 2, shs_w = mx ? Is / 32 : Is / 16;
#pragma omp parallel
    {
      std::vector<float> h(Imax), hhat(Imax);
      std::vector<uint8_t> hq_row(Imax), hsf_row(Imax / 16);
      std::vector<uint16_t> hb_row(Imax);
#pragma omp for schedule(dynamic, 4)
      for (int64_t t = 0; t < T; ++t) {
        expert_row(xhat.data() + t * H, Wg.data(), Wu.data(), Wd.data(), H, Is, a->ts_h, a,
                   a->act_mode, h.data(), hhat.data(), hq_row.data(), hsf_row.data(),
                   hb_row.data(), S.data() + t * H);
        if (a->act_mode != 1 && a->shq) std::memcpy(a->shq + t * shq_w, hq_row.data(), shq_w);
        if (a->act_mode != 1 && a->shsf) std::memcpy(a->shsf + t * shs_w, hsf_row.data(), shs_w);
        if (a->act_mode == 1 && a->shb) std::copy(hb_row.begin(), hb_row.begin() + Is, a->shb + t * Is);
      }
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int m = 0; m < H; ++m) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) acc = acc + w[t * k + j] * D[(int64_t)inv[t * k + j] * H + m];
      if (a->has_shared) acc = acc + S[t * H + m];
      a->y[t * H + m] = orc_f32_to_bf16(acc);
    }
  if (a->ids) std::copy(ids.begin(), ids.end(), a->ids);
  if (a->w) std::copy(w.begin(), w.end(), a->w);
  if (a->counts) std::copy(counts.begin(), counts.end(), a->counts);
  if (a->offsets) std::copy(offsets.begin(), offsets.end(), a->offsets);
  if (a->perm_src) std::copy(perm_src.begin(), perm_src.end(), a->perm_src);
  if (a->inv) std::copy(inv.begin(), inv.end(), a->inv);
  return 0;
}

// The same layer as a brute-force per-token loop: no permutation, every weight decoded at the
// point of use.  Used only to pin orc_moe_forward (the two must agree bit for bit).
int orc_moe_forward_bruteforce(const orc_moe_args* a) {
  const int64_t T = a->T;
  const int H = a->H, I = a->I, E = a->E, k = a->k;
  if (T == 0) return 0;
  std::vector<int32_t> ids(T * k);
  std::vector<float> w(T * k);
  orc_router_ex(a->logits, T, E, k, a->router_mode, a->router_bias, ids.data(), w.data());
  const int Imax = std::max(I, a->I_shared);
  std::vector<float> xr(H), h(Imax), hhat(Imax), d(H), acc(H);
  std::vector<uint8_t> hq_row(Imax / 2), hsf_row(Imax / 16);
  const int mode = a->act_mode;
  auto wval = [mode](const orc_expert& ex, int mat, int64_t row, int64_t col, int64_t K) {
    uint8_t byte = ex.codes[mat][row * (K / 2) + col / 2];
    uint8_t code = (col & 1) ? (byte >> 4) : (byte & 15);
    if (mode == 2)  // MXFP4: E8M0 per 32, no tensor scale
      return orc_e2m1_decode(code) * orc_e8m0_decode(ex.sf[mat][row * (K / 32) + col / 32]);
    return (orc_e2m1_decode(code) * orc_e4m3_decode(ex.sf[mat][row * (K / 16) + col / 16])) *
           ex.ts[mat];
  };
  auto run_expert = [&](const orc_expert& ex, int Ie) {
    for (int n = 0; n < Ie; ++n) {
      float g = 0.0f, u = 0.0f;
      if (a->act_kind != 1)
        for (int c = 0; c < H; ++c) g = g + xr[c] * wval(ex, 0, n, c, H);
      for (int c = 0; c < H; ++c) u = u + xr[c] * wval(ex, 1, n, c, H);
      h[n] = activation(g, u, a);
    }
    if (a->act_mode == 1) {              // W4A16: h in BF16
      for (int n = 0; n < Ie; ++n) hhat[n] = orc_bf16_to_f32(orc_f32_to_bf16(h[n]));
    } else if (a->act_mode == 2) {       // W4A8: h in MXFP8, block by block
      for (int b = 0; b < Ie / 32; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(h[b * 32 + i]));
        const float X = orc_e8m0_decode(orc_mx_scale(amax, 8));
        for (int i = 0; i < 32; ++i)
          hhat[b * 32 + i] = orc_e4m3_decode(orc_e4m3_encode(h[b * 32 + i] / X)) * X;
      }
    } else {
      for (int b = 0; b < Ie / 16; ++b) {  // requantise block by block, then decode
        quant_block16(h.data() + b * 16, a->ts_h, hq_row.data() + b * 8, hsf_row.data() + b);
        float s = orc_e4m3_decode(hsf_row[b]);
        for (int i = 0; i < 16; ++i) {
          uint8_t byte = hq_row[b * 8 + i / 2];
          uint8_t code = (i & 1) ? (byte >> 4) : (byte & 15);
          hhat[b * 16 + i] = (orc_e2m1_decode(code) * s) * a->ts_h;
        }
      }
    }
    for (int m = 0; m < H; ++m) {
      float s = 0.0f;
      for (int n = 0; n < Ie; ++n) s = s + hhat[n] * wval(ex, 2, m, n, Ie);
      d[m] = s;
    }
  };
  for (int64_t t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) {
      if (a->act_mode == 1) {
        xr[c] = orc_bf16_to_f32(a->x_bf16[t * H + c]);
        continue;
      }
      if (a->act_mode == 2) {  // MXFP8 of the token's row, block by block
        if (c % 32 == 0) {
          float amax = 0.0f;
          for (int i = 0; i < 32; ++i)
            amax = std::max(amax, std::fabs(orc_bf16_to_f32(a->x_bf16[t * H + c + i])));
          const float X = orc_e8m0_decode(orc_mx_scale(amax, 8));
          for (int i = 0; i < 32; ++i)
            xr[c + i] = orc_e4m3_decode(orc_e4m3_encode(orc_bf16_to_f32(a->x_bf16[t * H + c + i]) / X)) * X;
        }
        continue;
      }
      uint8_t byte = a->xq[t * (H / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      xr[c] = (orc_e2m1_decode(code) * orc_e4m3_decode(a->xsf[t * (H / 16) + c / 16])) * a->ts_a;
    }
    for (int m = 0; m < H; ++m) acc[m] = 0.0f;
    for (int j = 0; j < k; ++j) {
      run_expert(a->experts[ids[t * k + j]], I);
      for (int m = 0; m < H; ++m) acc[m] = acc[m] + w[t * k + j] * d[m];
    }
    if (a->has_shared) {
      run_expert(a->experts[E], a->I_shared);
      for (int m = 0; m < H; ++m) acc[m] = acc[m] + d[m];
    }
    for (int m = 0; m < H; ++m) a->y[t * H + m] = orc_f32_to_bf16(acc[m]);
  }
  return 0;
}

}  // extern "C"
