// NVFP4 quantisers: activations (one tensor scale, then per-16 blocks), expert weights (per expert
// and matrix, packed for the grouped GEMM), the export of packed weights back to the canonical
// layout, and the FP32 -> BF16 output rounding.
//
// Quantisation rule ("nvfp4-megamoe-kernel compare pre-b1...master", section "7. NVFP4
// Quantization": tensor scale max|x| / (6 * 448); block scales E4M3 over 16 elements, codes E2M1,
// section "NVFP4 throughout"): ts = amax / 2688, sf = E4M3((block_max / 6) / ts), code =
// E2M1(x / (decode(sf) * ts)), round to nearest even, IEEE FP32 division (no fast math).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxAmaxBlocks = 1024;

// Pass 1: max |x| over the whole tensor (BF16 magnitudes compare as their bit patterns), with a
// last-block reduction that writes ts = amax / 2688 and re-arms the block counter.  Optionally
// zero-fills `zero` (the FP32 output accumulator of the layer) on the way.  With ts_in (input
// already quantised, nvec = 0) the last block takes that tensor scale over instead.
__global__ void __launch_bounds__(kThreads) act_amax_kernel(const uint4* __restrict__ x,
                                                           int64_t nvec, WsHeader* hdr,
                                                           uint32_t* partials, float* ts_out,
                                                           float4* zero, int64_t nzero4,
                                                           const float* ts_in) {
  __shared__ uint32_t red[32];
  __shared__ bool is_last;
  griddep_wait();
  griddep_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t m = 0;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 4
  for (; i < nvec; i += stride) m = max(m, abs_bf16_max8(__ldg(x + i)));
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nzero4; j += stride)
    zero[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) {
    partials[blockIdx.x] = m;
    __threadfence();
    const uint32_t prev = atomicAdd(&hdr->counter, 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  uint32_t v = 0;
  for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x)
    v = max(v, __ldcg(partials + b));
  __syncthreads();
  v = block_max_u32(v, red);
  if (threadIdx.x == 0) {
    float ts;
    if (ts_in) {
      ts = *ts_in;
      if (!(ts >= 0.0f && ts <= 3.402823466e38f)) set_status(&hdr->status, MOE_ERR_NONFINITE);
    } else {
      if (v >= 0x7F80u) set_status(&hdr->status, MOE_ERR_NONFINITE);
      ts = __fdiv_rn(bf16_bits_to_f32(v), 2688.0f);
    }
    hdr->ts = ts;
    if (ts_out) *ts_out = ts;
    hdr->counter = 0u;
  }
}

// Pass 2: one thread per 16-element block: 32 bytes in, 8 code bytes and 1 scale byte out.
__global__ void __launch_bounds__(kThreads) act_encode_kernel(const uint4* __restrict__ x,
                                                             int64_t nblk,
                                                             const float* __restrict__ ts_ptr,
                                                             uint2* __restrict__ codes,
                                                             uint8_t* __restrict__ sf) {
  griddep_wait();
  griddep_launch();
  const float ts = *ts_ptr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += stride) {
    encode_bf16_block16(x, b, ts, codes, sf);
  }
}

// ---- weights ----

struct WeightSrc {
  const uint16_t* routed[3];  // gate [E,I,H], up [E,I,H], down [E,H,I]
  const uint16_t* shared[3];  // [Is,H], [Is,H], [H,Is] or null
  int E, H, I, Is;
  int gated;                  // 0: non-gated experts (ReLU2), no gate matrix to read or pack
};

__device__ __forceinline__ const uint16_t* matrix_ptr(const WeightSrc& w, int slot, int m,
                                                      int64_t per) {
  return slot < w.E ? w.routed[m] + (int64_t)slot * per : w.shared[m];
}

// Row of the gate (m=0) or up (m=1) row n inside the 16-interleaved w13 layout (gated experts),
// or of up row n in the up-only w13 layout (non-gated experts).
__host__ __device__ __forceinline__ int64_t w13_row(int64_t n, int m, int gated) {
  return gated ? (n >> 4) * 32 + (m ? 16 : 0) + (n & 15) : n;
}

// max |W| per (slot, matrix) as BF16 magnitude bits, atomically max-ed into amax_bits[slot*4+m].
__global__ void __launch_bounds__(kThreads) weight_amax_kernel(WeightSrc w, uint32_t* amax_bits) {
  __shared__ uint32_t red[32];
  const int mi = blockIdx.y;
  const int slot = mi / 3, m = mi % 3;
  if (m == 0 && !w.gated) return;   // no gate matrix: its tensor scale stays 0
  const int64_t per = (int64_t)(slot < w.E ? w.I : w.Is) * w.H;
  const uint4* src = reinterpret_cast<const uint4*>(matrix_ptr(w, slot, m, per));
  const int64_t nvec = per / 8;
  uint32_t v = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x)
    v = max(v, abs_bf16_max8(__ldg(src + i)));
  v = block_max_u32(v, red);
  if (threadIdx.x == 0) atomicMax(amax_bits + slot * 4 + m, v);
}

__global__ void weight_ts_kernel(uint32_t* amax_bits_then_ts, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const float amax = bf16_bits_to_f32(amax_bits_then_ts[i]);
    reinterpret_cast<float*>(amax_bits_then_ts)[i] = __fdiv_rn(amax, 2688.0f);
  }
}

struct WeightDst {
  uint8_t* w13;     // [Et][2I/128][H/256][block] ([Et][I/128][H/256][block] when not gated)
  uint8_t* w2;      // [Et][H/128][I/256][block]
  const float* ts;  // [Et][4]
  int64_t w13_per_e, w2_per_e;
  int gated;
  int H, I;         // the packed (256-multiple) widths: K of the packed blocks
};

// One thread per 16-element block of one matrix row: quantise and store into the packed layout.
__global__ void __launch_bounds__(kThreads) weight_encode_kernel(WeightSrc w, WeightDst d) {
  const int mi = blockIdx.y;
  const int slot = mi / 3, m = mi % 3;
  if (m == 0 && !w.gated) return;
  const int Iw = slot < w.E ? w.I : w.Is;   // this expert's intermediate size
  const int64_t per = (int64_t)Iw * w.H;
  const int64_t K = m < 2 ? w.H : Iw;
  const int64_t nblk = per / 16;
  const uint16_t* src = matrix_ptr(w, slot, m, per);
  const float ts = d.ts[slot * 4 + m];
  const int64_t Kp = m < 2 ? d.H : d.I;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = b / (K / 16), kb = b % (K / 16);
    const uint4* p = reinterpret_cast<const uint4*>(src + n * K + kb * 16);
    const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = bf16_bits_to_f32(wv[i] & 0xFFFFu);
      f[2 * i + 1] = bf16_bits_to_f32(wv[i] >> 16);
    }
    uint32_t lo, hi, s;
    quant_block16(f, ts, lo, hi, s);
    uint8_t* base = m < 2 ? d.w13 + slot * d.w13_per_e : d.w2 + slot * d.w2_per_e;
    const int64_t r = m < 2 ? w13_row(n, m, d.gated) : n;
    *reinterpret_cast<uint2*>(base + packed_code_offset(r, kb, Kp)) = make_uint2(lo, hi);
    base[packed_sf_offset(r, kb, Kp)] = (uint8_t)s;
  }
}

// MXFP4 weights (the W4A8 layer): one thread per 32-element block of one matrix row.  Codes go to
// the same packed positions as NVFP4 codes; the block's E8M0 scale byte to the block's scale
// area at row * 8 + (32-block within the 256-wide K stage).
__host__ __device__ __forceinline__ size_t packed_mx_sf_offset(int64_t n, int64_t kb32, int64_t K) {
  const int64_t kst = K / 256, r = n & 127;
  const int64_t blk = (n >> 7) * kst + kb32 / 8;
  return (size_t)(blk * kTileBlockBytes + kTileBytes + r * 8 + (kb32 & 7));
}

__global__ void __launch_bounds__(kThreads) weight_encode_mx_kernel(WeightSrc w, WeightDst d) {
  const int mi = blockIdx.y;
  const int slot = mi / 3, m = mi % 3;
  if (m == 0 && !w.gated) return;
  const int Iw = slot < w.E ? w.I : w.Is;   // this expert's intermediate size
  const int64_t per = (int64_t)Iw * w.H;
  const int64_t K = m < 2 ? w.H : Iw;
  const int64_t nblk = per / 32;
  const uint16_t* src = matrix_ptr(w, slot, m, per);
  const int64_t Kp = m < 2 ? d.H : d.I;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = b / (K / 32), kb = b % (K / 32);
    const uint4* p = reinterpret_cast<const uint4*>(src + n * K + kb * 32);
    float f[32];
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(p + q);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[8 * q + 2 * i] = bf16_bits_to_f32(wv[i] & 0xFFFFu);
        f[8 * q + 2 * i + 1] = bf16_bits_to_f32(wv[i] >> 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const uint32_t sb = mx_scale_byte(amax, 2);
    uint32_t words[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      words[q] = e2m1x8(mx_unscale(f[8 * q], sb), mx_unscale(f[8 * q + 1], sb),
                        mx_unscale(f[8 * q + 2], sb), mx_unscale(f[8 * q + 3], sb),
                        mx_unscale(f[8 * q + 4], sb), mx_unscale(f[8 * q + 5], sb),
                        mx_unscale(f[8 * q + 6], sb), mx_unscale(f[8 * q + 7], sb));
    uint8_t* base = m < 2 ? d.w13 + slot * d.w13_per_e : d.w2 + slot * d.w2_per_e;
    const int64_t r = m < 2 ? w13_row(n, m, d.gated) : n;
    *reinterpret_cast<uint2*>(base + packed_code_offset(r, 2 * kb, Kp)) =
        make_uint2(words[0], words[1]);
    *reinterpret_cast<uint2*>(base + packed_code_offset(r, 2 * kb + 1, Kp)) =
        make_uint2(words[2], words[3]);
    base[packed_mx_sf_offset(r, kb, Kp)] = (uint8_t)sb;
  }
}

__global__ void weight_ts_one_kernel(float* ts, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) ts[i] = 1.0f;
}

// Canonical MXFP4 export: codes [N, K/2], E8M0 scales [N, K/32].
__global__ void __launch_bounds__(kThreads) weight_export_mx_kernel(WeightDst d, int slot, int m,
                                                                   int64_t N, int64_t K,
                                                                   uint8_t* codes, uint8_t* sf,
                                                                   float* ts) {
  const int64_t nblk = N * K / 16;
  const int64_t Kp = m < 2 ? d.H : d.I;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = b / (K / 16), kb = b % (K / 16);
    const uint8_t* base = m < 2 ? d.w13 + slot * d.w13_per_e : d.w2 + slot * d.w2_per_e;
    const int64_t r = m < 2 ? w13_row(n, m, d.gated) : n;
    *reinterpret_cast<uint2*>(codes + n * (K / 2) + kb * 8) =
        *reinterpret_cast<const uint2*>(base + packed_code_offset(r, kb, Kp));
    if ((kb & 1) == 0) sf[n * (K / 32) + kb / 2] = base[packed_mx_sf_offset(r, kb / 2, Kp)];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts = d.ts[slot * 4 + m];
}

__global__ void __launch_bounds__(kThreads) weight_export_kernel(WeightDst d, int slot, int m,
                                                                int64_t N, int64_t K,
                                                                uint8_t* codes, uint8_t* sf,
                                                                float* ts) {
  const int64_t nblk = N * K / 16;
  const int64_t Kp = m < 2 ? d.H : d.I;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = b / (K / 16), kb = b % (K / 16);
    const uint8_t* base = m < 2 ? d.w13 + slot * d.w13_per_e : d.w2 + slot * d.w2_per_e;
    const int64_t r = m < 2 ? w13_row(n, m, d.gated) : n;
    const uint2 c = *reinterpret_cast<const uint2*>(base + packed_code_offset(r, kb, Kp));
    const uint8_t s = base[packed_sf_offset(r, kb, Kp)];
    *reinterpret_cast<uint2*>(codes + n * (K / 2) + kb * 8) = c;
    sf[n * (K / 16) + kb] = s;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts = d.ts[slot * 4 + m];
}

__global__ void __launch_bounds__(kThreads) finalize_kernel(const float4* __restrict__ acc,
                                                           uint2* __restrict__ y, int64_t n4) {
  griddep_wait();
  griddep_launch();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = __ldcs(acc + i);
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    y[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

// y[t] = bf16( sum_{j<k} o[inv[t*k+j]] (+ o[T*k + t] for the shared expert) ), summed in slot
// order; o holds each assignment's router-weighted expert output in FP32.
__global__ void __launch_bounds__(kThreads) finalize_gather_kernel(const float4* __restrict__ o,
                                                                  const int32_t* __restrict__ inv,
                                                                  int T, int k, int H4,
                                                                  int shared, uint2* __restrict__ y,
                                                                  int32_t* plan_flag) {
  griddep_wait();
  griddep_launch();
  // the decode GEMM of this call has completed (the wait above), so nothing reads the plan-ready
  // flag any more: lower it for the next call (its prologue lowers it again before the next GEMM
  // may launch)
  if (plan_flag && blockIdx.x == 0 && threadIdx.x == 0) *plan_flag = 0;
  const int64_t n = (int64_t)T * H4;
  const int64_t R = (int64_t)T * k;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / H4, m = i - t * H4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // eight slots at a time: their row indices, then their rows, then the in-order additions
    // (two dependent memory round trips per group instead of two per slot)
    for (int j0 = 0; j0 < k; j0 += 8) {
      int row[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) row[u] = j0 + u < k ? __ldg(inv + t * k + j0 + u) : 0;
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = j0 + u < k ? __ldcg(o + (int64_t)row[u] * H4 + m) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < k) {
          acc.x = __fadd_rn(acc.x, v[u].x);
          acc.y = __fadd_rn(acc.y, v[u].y);
          acc.z = __fadd_rn(acc.z, v[u].z);
          acc.w = __fadd_rn(acc.w, v[u].w);
        }
      }
    }
    if (shared) {
      const float4 v = __ldcg(o + (R + t) * H4 + m);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc.z, acc.w);
    y[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

// Expert-ordered copy of the quantised activations: 16-byte code vectors, then 4-scale words into
// the 32x4x4 arrangement of the GEMM tiles (see launch_permute_rows).
// Activation encode straight into expert order (batches planned before they are encoded): one
// thread per 16-element block of x quantises it once and writes it in token order and into each
// of the token's expert-ordered rows - its codes into xq_perm, its scale byte into the
// 32x4x4 arrangement of the GEMM's A-operand scales (tile = the segment's first tile + row/128).
__global__ void __launch_bounds__(kThreads) act_encode_perm_kernel(
    const uint4* __restrict__ x, int T, int H, int k, int E, int shared, int Rt,
    const float* __restrict__ ts_ptr, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_start, uint2* __restrict__ codes, uint8_t* __restrict__ sf,
    uint8_t* __restrict__ xq_perm, uint8_t* __restrict__ xsf_tiles, int32_t* status) {
  griddep_wait();
  griddep_launch();
  const float ts = *ts_ptr;
  const int nkb = H / 16, wpr = H / 64;
  const int64_t nblk = (int64_t)T * nkb;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nblk; u += stride) {
    const int t = (int)(u / nkb), b = (int)(u - (int64_t)t * nkb);
    uint32_t lo, hi, s8;
    quant_bf16_block16(x, u, ts, lo, hi, s8);
    if (codes) {   // the token-order copy (read only by the debug copies)
      codes[u] = make_uint2(lo, hi);
      sf[u] = (uint8_t)s8;
    }
    for (int j = 0; j <= k; ++j) {
      int p, seg;
      if (j < k) {
        seg = __ldg(ids + (int64_t)t * k + j);
        p = __ldg(inv + (int64_t)t * k + j);
      } else {
        if (!shared) break;
        seg = E;
        p = T * k + t;   // the shared expert's rows follow the routed ones, in token order
      }
      if (seg < 0 || seg > E || p < 0 || p >= Rt) {
        set_status(status, MOE_ERR_INVALID_ARG);
        continue;
      }
      const int r = p - __ldg(offsets + seg);
      if (r < 0) {
        set_status(status, MOE_ERR_INVALID_ARG);
        continue;
      }
      const int64_t tile = __ldg(tile_start + seg) + (r >> 7);
      const int rr = r & 127;
      *reinterpret_cast<uint2*>(xq_perm + (size_t)p * (H / 2) + (size_t)b * 8) = make_uint2(lo, hi);
      xsf_tiles[(tile * wpr + b / 4) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (b & 3)] = (uint8_t)s8;
    }
  }
}

// ---- RMSNorm + NVFP4 quantisation (the producer feeding the activation quantiser) ----
// Scratch: [0] the tensor's max |y| as float bits, [1] the finished-block count, [2] the tensor
// scale, [4 .. 4+rows) each row's 1/rms.  Every FP32 operation is an explicit round-to-nearest
// intrinsic, so nothing is contracted into a fused multiply-add.

// Pass 1: one warp per row (rows taken in turn).  The definition of the mean square is the exact
// sum of the squares rounded once to FP32; this kernel forms it in FP32 in its own order, which
// keeps the loads coalesced: chunks of 8 elements summed left to right, then a balanced tree over
// the chunk index (zero-padded to a power of two).  In step j the warp loads chunks
// 32j .. 32j+31 (lane l: chunk 32j + l, one coalesced 512-byte run) and its xor butterfly forms
// the tree's first five levels over them; the J step sums then form the remaining levels, in
// registers.  Every term is non-negative, so the relative error of the sum is at most
// (7 + 5 + log2 J) * 2^-24 (at most 18 * 2^-24 for 16384 columns).
// 1/rms = 1/sqrt(mean + eps), y = (x * r) * gamma;
// each block keeps its max |y|, and the block that finishes last turns the tensor max into the
// tensor scale.
template <int J>
__global__ void __launch_bounds__(kThreads) rmsnorm_amax_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ gamma, float eps, int64_t rows,
    int cols, uint32_t* __restrict__ scratch, float* __restrict__ rrms, int32_t* status) {
  __shared__ uint32_t red[32];
  __shared__ bool is_last;
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int nchunk = cols / 8;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  uint32_t m = 0u;
  for (int64_t row = wid; row < rows; row += nwarps) {
    const uint4* xr = x + row * nchunk;
    float part[J];
    // eight steps' loads in flight at a time, then their chunk sums and butterflies
#pragma unroll
    for (int j0 = 0; j0 < J; j0 += 8) {
      uint4 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = (j0 + u) * 32 + lane;
        q[u] = (j0 + u < J && c < nchunk) ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= J) break;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
        float v = bf16_bits_to_f32(w[0] & 0xFFFFu);
        float sq = __fmul_rn(v, v);
#pragma unroll
        for (int i = 1; i < 8; ++i) {
          v = bf16_bits_to_f32((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
          sq = __fadd_rn(sq, __fmul_rn(v, v));
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
        part[j0 + u] = sq;
      }
    }
#pragma unroll
    for (int width = 1; width < J; width *= 2)
#pragma unroll
      for (int i = 0; i < J; i += 2 * width) part[i] = __fadd_rn(part[i], part[i + width]);
    const float sum = part[0];
    const float ms = __fdiv_rn(sum, (float)cols);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    if (lane == 0) {
      reinterpret_cast<float*>(scratch)[4 + row] = r;
      if (rrms) rrms[row] = r;
    }
#pragma unroll
    for (int j0 = 0; j0 < J; j0 += 8) {
      uint4 q[8], gm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = (j0 + u) * 32 + lane;
        const bool in = j0 + u < J && c < nchunk;
        q[u] = in ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
        gm[u] = in ? __ldg(gamma + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
        const uint32_t gw[4] = {gm[u].x, gm[u].y, gm[u].z, gm[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // padding chunks are zero and leave the max unchanged
          const float y0 = __fmul_rn(__fmul_rn(bf16_bits_to_f32(w[i] & 0xFFFFu), r),
                                     bf16_bits_to_f32(gw[i] & 0xFFFFu));
          const float y1 = __fmul_rn(__fmul_rn(bf16_bits_to_f32(w[i] >> 16), r),
                                     bf16_bits_to_f32(gw[i] >> 16));
          m = max(m, max(__float_as_uint(fabsf(y0)), __float_as_uint(fabsf(y1))));
        }
      }
    }
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) {
    atomicMax(scratch, m);   // non-negative floats order like their bit patterns (NaN above inf)
    __threadfence();
    is_last = atomicAdd(scratch + 1, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;
  __threadfence();
  const uint32_t amax = atomicAdd(scratch, 0u);
  if (amax >= 0x7F800000u) set_status(status, MOE_ERR_NONFINITE);
  reinterpret_cast<float*>(scratch)[2] = __fdiv_rn(__uint_as_float(amax), 2688.0f);
  scratch[0] = 0u;
  scratch[1] = 0u;
}

// Pass 2, one thread per 16-element block: y recomputed exactly as in pass 1, then encoded.
__global__ void __launch_bounds__(kThreads) rmsnorm_encode_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ gamma, int64_t rows, int cols,
    const uint32_t* __restrict__ scratch, uint2* __restrict__ codes, uint8_t* __restrict__ sf,
    float* ts_out) {
  griddep_wait();
  griddep_launch();
  const float ts = __ldcg(reinterpret_cast<const float*>(scratch) + 2);
  const float* rr = reinterpret_cast<const float*>(scratch) + 4;
  const int bpr = cols / 16;
  const int64_t nblk = rows * bpr;
  if (blockIdx.x == 0 && threadIdx.x == 0 && ts_out) *ts_out = ts;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += stride) {
    const int64_t row = b / bpr;
    const int cb = (int)(b - row * bpr);
    const float r = __ldcg(rr + row);
    const uint4 q0 = __ldg(x + 2 * b), q1 = __ldg(x + 2 * b + 1);
    const uint4 g0 = __ldg(gamma + 2 * cb), g1 = __ldg(gamma + 2 * cb + 1);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float y[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      y[2 * j] = __fmul_rn(__fmul_rn(bf16_bits_to_f32(w[j] & 0xFFFFu), r),
                           bf16_bits_to_f32(gw[j] & 0xFFFFu));
      y[2 * j + 1] = __fmul_rn(__fmul_rn(bf16_bits_to_f32(w[j] >> 16), r),
                               bf16_bits_to_f32(gw[j] >> 16));
    }
    uint32_t lo, hi, s8;
    quant_block16(y, ts, lo, hi, s8);
    codes[b] = make_uint2(lo, hi);
    sf[b] = (uint8_t)s8;
  }
}

__global__ void __launch_bounds__(kThreads) permute_rows_kernel(
    const uint4* __restrict__ xq, const uint32_t* __restrict__ xsf, int T, int H, int Rt, int E,
    const int32_t* __restrict__ perm_src, const int32_t* __restrict__ perm_seg,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_start,
    uint4* __restrict__ xq_perm, uint8_t* __restrict__ xsf_tiles, int32_t* status) {
  griddep_wait();
  griddep_launch();
  const int vpr = H / 32, wpr = H / 64;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t nvec = (int64_t)Rt * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const int64_t p = i / vpr;
    const int v = (int)(i - p * vpr);
    const int t = __ldg(perm_src + p);
    if (t < 0 || t >= T) {
      set_status(status, MOE_ERR_INVALID_ARG);
      continue;
    }
    xq_perm[p * vpr + v] = __ldg(xq + (int64_t)t * vpr + v);
  }
  const int64_t nw = (int64_t)Rt * wpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw; i += stride) {
    const int64_t p = i / wpr;
    const int wd = (int)(i - p * wpr);
    const int t = __ldg(perm_src + p);
    const int e = __ldg(perm_seg + p);
    if (t < 0 || t >= T || e < 0 || e > E) {
      set_status(status, MOE_ERR_INVALID_ARG);
      continue;
    }
    const int r = (int)(p - __ldg(offsets + e));
    if (r < 0) {
      set_status(status, MOE_ERR_INVALID_ARG);
      continue;
    }
    const int64_t tile = __ldg(tile_start + e) + (r >> 7);
    const int rr = r & 127;
    *reinterpret_cast<uint32_t*>(xsf_tiles + (tile * wpr + wd) * 512 + (rr & 31) * 16 + (rr >> 5) * 4) =
        __ldg(xsf + (int64_t)t * wpr + wd);
  }
}

// BF16 token rows into expert order (the W4A16 layer's A operand): 16-byte vectors.
__global__ void __launch_bounds__(kThreads) permute_rows_bf16_kernel(
    const uint4* __restrict__ x, int T, int vpr, int Rt, const int32_t* __restrict__ perm_src,
    uint4* __restrict__ xb_perm, int32_t* status) {
  griddep_wait();
  griddep_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t nvec = (int64_t)Rt * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const int64_t p = i / vpr;
    const int v = (int)(i - p * vpr);
    const int t = __ldg(perm_src + p);
    if (t < 0 || t >= T) {
      set_status(status, MOE_ERR_INVALID_ARG);
      continue;
    }
    xb_perm[p * vpr + v] = __ldg(x + (int64_t)t * vpr + v);
  }
}

// The W4A8 layer's activations: one thread per 32-element block of x: MXFP8 (E8M0 scale for E4M3
// elements, codes rounded to nearest even and saturated), written in token order (codes [T, H],
// scales [T, H/32]) and, decoded back to BF16 (exact: 4 significant bits times a power of two),
// into each of the token's expert-ordered rows of xb_perm [Rt, H] (the GEMM's A operand).
__global__ void __launch_bounds__(kThreads) act_mx_encode_perm_kernel(
    const uint4* __restrict__ x, int T, int H, int k, int shared, int Rt,
    const int32_t* __restrict__ inv, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    uint4* __restrict__ xb_perm, int32_t* status) {
  griddep_wait();
  griddep_launch();
  const int nkb = H / 32;
  const int64_t nblk = (int64_t)T * nkb;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nblk; u += stride) {
    const int t = (int)(u / nkb), b = (int)(u - (int64_t)t * nkb);
    float f[32];
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(x + 4 * u + q);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[8 * q + 2 * i] = bf16_bits_to_f32(wv[i] & 0xFFFFu);
        f[8 * q + 2 * i + 1] = bf16_bits_to_f32(wv[i] >> 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    if (!(amax <= 3.402823466e38f)) set_status(status, MOE_ERR_NONFINITE);
    const uint32_t sb = mx_scale_byte(amax, 8);
    const float X = e8m0_to_f32(sb);
    uint32_t cw[8];
    uint4 out[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t c = 0u;
#pragma unroll
      for (int j = 0; j < 4; j += 2)
        c |= f32_to_e4m3x2(mx_unscale(f[4 * i + j], sb), mx_unscale(f[4 * i + j + 1], sb)) << (8 * j);
      cw[i] = c;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t ow[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c2 = (cw[2 * q + i / 2] >> (16 * (i & 1))) & 0xFFFFu;
        const float2 v = e4m3x2_to_f32x2(c2);
        const __nv_bfloat162 bb = __floats2bfloat162_rn(v.x * X, v.y * X);
        ow[i] = *reinterpret_cast<const uint32_t*>(&bb);
      }
      out[q] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
    uint4* cdst = reinterpret_cast<uint4*>(codes + u * 32);
    cdst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    cdst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    sf[u] = (uint8_t)sb;
    for (int j = 0; j <= k; ++j) {
      int p;
      if (j < k) {
        p = __ldg(inv + (int64_t)t * k + j);
      } else {
        if (!shared) break;
        p = T * k + t;
      }
      if (p < 0 || p >= Rt) {
        set_status(status, MOE_ERR_INVALID_ARG);
        continue;
      }
      uint4* dst = xb_perm + ((size_t)p * H + (size_t)b * 32) / 8;
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = out[q];
    }
  }
}

int grid_for(int64_t work, int per_block, int cap) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

WeightDst make_dst(const WeightLayout& L, uint8_t* wbuf) {
  WeightDst d;
  d.w13 = wbuf + L.w13;
  d.w2 = wbuf + L.w2;
  d.ts = reinterpret_cast<const float*>(wbuf + L.ts);
  d.w13_per_e = (int64_t)L.w13_per_e;
  d.w2_per_e = (int64_t)L.w2_per_e;
  d.gated = L.gated ? 1 : 0;
  d.H = L.H;
  d.I = L.I;
  return d;
}

}  // namespace

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

cudaError_t launch_act_amax(const void* x, int64_t rows, int64_t cols, float* ts, WsHeader* hdr,
                            uint32_t* partials, float* zero_buf, int64_t zero_floats,
                            cudaStream_t s, const float* ts_in) {
  const int64_t nvec = ts_in ? 0 : rows * cols / 8;
  // sized for the larger of the two jobs: a caller that only zero-fills (rows = 0) still gets a
  // grid as wide as the fill
  const int g1 = grid_for(std::max(nvec, zero_floats / 4), kThreads * 8, kMaxAmaxBlocks);
  return launch_pdl(act_amax_kernel, dim3(g1), dim3(kThreads), 0, s,
                    reinterpret_cast<const uint4*>(x), nvec, hdr, partials, ts,
                    reinterpret_cast<float4*>(zero_buf), zero_floats / 4, ts_in);
}

cudaError_t launch_act_encode_perm(const void* x, int T, int H, int k, int E, int shared, int Rt,
                                   const float* ts, const int32_t* ids, const int32_t* inv,
                                   const int32_t* offsets, const int32_t* tile_start,
                                   uint8_t* codes, uint8_t* sf, uint8_t* xq_perm,
                                   uint8_t* xsf_tiles, int32_t* status, cudaStream_t s) {
  const int64_t nblk = (int64_t)T * H / 16;
  const int g = grid_for(nblk, kThreads, num_sms() * 16);
  return launch_pdl(act_encode_perm_kernel, dim3(g), dim3(kThreads), 0, s,
                    reinterpret_cast<const uint4*>(x), T, H, k, E, shared, Rt, ts, ids, inv,
                    offsets, tile_start, reinterpret_cast<uint2*>(codes), sf, xq_perm, xsf_tiles,
                    status);
}

cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t rows,
                                 int64_t cols, uint8_t* codes, uint8_t* sf, float* ts,
                                 float* rrms, uint32_t* scratch, int32_t* status, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(scratch, 0, 4 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  // lanes own J chunks each: the padded chunk count (a power of two >= 32) over 32 lanes
  const int nchunk = (int)(cols / 8);
  int J = 1;
  while (J * 32 < nchunk) J *= 2;
  const int g1 = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 8);
#define NVFP4MOE_RMS(JJ)                                                                      \
  e = launch_pdl(rmsnorm_amax_kernel<JJ>, dim3(g1), dim3(kThreads), 0, s,                      \
                 reinterpret_cast<const uint4*>(x), reinterpret_cast<const uint4*>(gamma), eps, \
                 rows, (int)cols, scratch, rrms, status)
  switch (J) {
    case 1: NVFP4MOE_RMS(1); break;
    case 2: NVFP4MOE_RMS(2); break;
    case 4: NVFP4MOE_RMS(4); break;
    case 8: NVFP4MOE_RMS(8); break;
    case 16: NVFP4MOE_RMS(16); break;
    case 32: NVFP4MOE_RMS(32); break;
    case 64: NVFP4MOE_RMS(64); break;
    default: return cudaErrorInvalidValue;
  }
#undef NVFP4MOE_RMS
  if (e != cudaSuccess) return e;
  const int64_t nblk = rows * cols / 16;
  return launch_pdl(rmsnorm_encode_kernel, dim3(grid_for(nblk, kThreads, num_sms() * 16)),
                    dim3(kThreads), 0, s, reinterpret_cast<const uint4*>(x),
                    reinterpret_cast<const uint4*>(gamma), rows, (int)cols,
                    (const uint32_t*)scratch, reinterpret_cast<uint2*>(codes), sf, ts);
}

cudaError_t launch_act_quant(const void* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                             float* ts, WsHeader* hdr, uint32_t* partials, float* zero_buf,
                             int64_t zero_floats, cudaStream_t s) {
  const int64_t n = rows * cols;
  cudaError_t e = launch_act_amax(x, rows, cols, ts, hdr, partials, zero_buf, zero_floats, s,
                                  nullptr);
  if (e != cudaSuccess) return e;
  const int64_t nblk = n / 16;
  const int g2 = grid_for(nblk, kThreads, num_sms() * 16);
  return launch_pdl(act_encode_kernel, dim3(g2), dim3(kThreads), 0, s,
                    reinterpret_cast<const uint4*>(x), nblk, (const float*)&hdr->ts,
                    reinterpret_cast<uint2*>(codes), sf);
}

cudaError_t launch_weight_quant(const moe_config& c, const WeightLayout& L, const void* wg,
                                const void* wu, const void* wd, const void* sg, const void* su,
                                const void* sd, uint8_t* wbuf, cudaStream_t s) {
  WeightSrc w;
  w.routed[0] = static_cast<const uint16_t*>(wg);
  w.routed[1] = static_cast<const uint16_t*>(wu);
  w.routed[2] = static_cast<const uint16_t*>(wd);
  w.shared[0] = static_cast<const uint16_t*>(sg);
  w.shared[1] = static_cast<const uint16_t*>(su);
  w.shared[2] = static_cast<const uint16_t*>(sd);
  w.E = c.num_experts;
  w.H = c.hidden;
  w.I = c.inter;
  w.Is = c.shared_inter > 0 ? c.shared_inter : c.inter;
  w.gated = L.gated ? 1 : 0;
  uint32_t* amax = reinterpret_cast<uint32_t*>(wbuf + L.ts);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * 4 * L.Et, s);
  if (e != cudaSuccess) return e;
  const int64_t per = (int64_t)h_width(c) * c.hidden;   // the largest matrix
  dim3 g1(grid_for(per / 8, kThreads * 8, 256), L.Et * 3);
  weight_amax_kernel<<<g1, kThreads, 0, s>>>(w, amax);
  weight_ts_kernel<<<(L.Et * 4 + 255) / 256, 256, 0, s>>>(amax, L.Et * 4);
  WeightDst d = make_dst(L, wbuf);
  if (c.flags & MOE_FLAG_ACT_MXFP8) {   // MXFP4: E8M0 per 32, no tensor scale (kept at 1)
    weight_ts_one_kernel<<<(L.Et * 4 + 255) / 256, 256, 0, s>>>(reinterpret_cast<float*>(amax),
                                                                 L.Et * 4);
    dim3 gm(grid_for(per / 32, kThreads, 4096), L.Et * 3);
    weight_encode_mx_kernel<<<gm, kThreads, 0, s>>>(w, d);
    return cudaGetLastError();
  }
  dim3 g2(grid_for(per / 16, kThreads, 4096), L.Et * 3);
  weight_encode_kernel<<<g2, kThreads, 0, s>>>(w, d);
  return cudaGetLastError();
}

cudaError_t launch_weight_export(const moe_config& c, const WeightLayout& L, const uint8_t* wbuf,
                                 int slot, int m, uint8_t* codes, uint8_t* sf, float* ts,
                                 cudaStream_t s) {
  WeightDst d = make_dst(L, const_cast<uint8_t*>(wbuf));
  const int64_t Iw = slot < c.num_experts ? c.inter : c.shared_inter;   // this expert's width
  const int64_t N = m < 2 ? Iw : c.hidden;
  const int64_t K = m < 2 ? c.hidden : Iw;
  if (c.flags & MOE_FLAG_ACT_MXFP8)
    weight_export_mx_kernel<<<grid_for(N * K / 16, kThreads, 4096), kThreads, 0, s>>>(
        d, slot, m, N, K, codes, sf, ts);
  else
    weight_export_kernel<<<grid_for(N * K / 16, kThreads, 4096), kThreads, 0, s>>>(
        d, slot, m, N, K, codes, sf, ts);
  return cudaGetLastError();
}

cudaError_t launch_finalize_gather(const float* o, const int32_t* inv, int T, int k, int H,
                                   int shared, void* y, cudaStream_t s, int32_t* plan_flag) {
  const int64_t n4 = (int64_t)T * (H / 4);
  return launch_pdl(finalize_gather_kernel, dim3(grid_for(n4, kThreads, num_sms() * 8)),
                    dim3(kThreads), 0, s, reinterpret_cast<const float4*>(o), inv, T, k, H / 4,
                    shared, reinterpret_cast<uint2*>(y), plan_flag);
}

cudaError_t launch_permute_rows(const uint8_t* xq, const uint8_t* xsf, int T, int H, int Rt,
                                int E, const int32_t* perm_src, const int32_t* perm_seg,
                                const int32_t* offsets, const int32_t* tile_start,
                                uint8_t* xq_perm, uint8_t* xsf_tiles, int32_t* status,
                                cudaStream_t s) {
  const int64_t work = (int64_t)Rt * (H / 32);
  return launch_pdl(permute_rows_kernel, dim3(grid_for(work, kThreads, num_sms() * 8)),
                    dim3(kThreads), 0, s, reinterpret_cast<const uint4*>(xq),
                    reinterpret_cast<const uint32_t*>(xsf), T, H, Rt, E, perm_src, perm_seg,
                    offsets, tile_start, reinterpret_cast<uint4*>(xq_perm), xsf_tiles, status);
}

cudaError_t launch_permute_rows_bf16(const void* x, int T, int H, int Rt, const int32_t* perm_src,
                                     void* xb_perm, int32_t* status, cudaStream_t s) {
  const int vpr = H / 8;
  const int64_t work = (int64_t)Rt * vpr;
  return launch_pdl(permute_rows_bf16_kernel, dim3(grid_for(work, kThreads, num_sms() * 8)),
                    dim3(kThreads), 0, s, reinterpret_cast<const uint4*>(x), T, vpr, Rt, perm_src,
                    reinterpret_cast<uint4*>(xb_perm), status);
}

cudaError_t launch_act_mx_encode_perm(const void* x, int T, int H, int k, int shared, int Rt,
                                      const int32_t* inv, uint8_t* codes, uint8_t* sf,
                                      void* xb_perm, int32_t* status, cudaStream_t s) {
  const int64_t nblk = (int64_t)T * H / 32;
  return launch_pdl(act_mx_encode_perm_kernel, dim3(grid_for(nblk, kThreads, num_sms() * 16)),
                    dim3(kThreads), 0, s, reinterpret_cast<const uint4*>(x), T, H, k, shared, Rt,
                    inv, codes, sf, reinterpret_cast<uint4*>(xb_perm), status);
}

cudaError_t launch_finalize(const float* yacc, void* y, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;
  return launch_pdl(finalize_kernel, dim3(grid_for(n4, kThreads, num_sms() * 8)), dim3(kThreads),
                    0, s, reinterpret_cast<const float4*>(yacc), reinterpret_cast<uint2*>(y), n4);
}

}  // namespace nvfp4moe
