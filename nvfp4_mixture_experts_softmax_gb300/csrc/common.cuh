// Device helpers shared by the NVFP4 MoE kernels (sm_103a): format conversions through the PTX
// cvt instructions, mbarrier / TMA / tcgen05 wrappers, and bounded waits.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4_moe.h"

namespace nvfp4moe {

// Programmatic dependent launch: a kernel launched with the programmatic-serialization attribute
// may start while its predecessor in the stream is still running.  Each kernel of the layer
// calls griddep_wait() before its first access to global memory (so every read sees the
// predecessor's writes and no write races a read of the predecessor) and griddep_launch() to
// let its own successor start launching.  Both are no-ops for an ordinary launch.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Device status word: the first error wins.
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------------------------
// Formats.  E4M3 and E2M1 conversions use the documented PTX cvt instructions, which round to
// nearest even and, with .satfinite, clamp finite overflow (and infinities) to the largest
// finite value.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// Two FP32 values -> two E4M3 codes in the low 16 bits, the first value in the low byte.
__device__ __forceinline__ uint32_t f32_to_e4m3x2(float v0, float v1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v1), "f"(v0));
  return r;
}

// Two E4M3 codes (low byte first) -> two FP32 values (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t b2) {
  uint32_t h2;
  const uint16_t in = (uint16_t)(b2 & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Eight FP32 values -> eight E2M1 codes in one word, element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t r;
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// NVFP4 quantisation of one 16-element block with tensor scale ts.
//   sf = E4M3((max|x| / 6) / ts); S = decode(sf) * ts; code_i = E2M1(x_i / S)
// with IEEE FP32 division and multiplication in that order; a zero block or a zero S gives scale
// byte 0 and all-zero codes.
// x / S rounded to nearest even, from r = RN(1/S): q0 = RN(x*r) is within 1.5 ulp of x/S (the
// reciprocal and the product each round once), the residual x - q0*S is formed by one fma, and
// q1 = RN(q0 + residual*r) is returned.  The quotient only decides an E2M1 code, so what has to
// be right is on which side of each rounding boundary b (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5)
// RN(x/S) lies, and whether it equals b.  For every one of the 2^23 FP32 significands of S and
// every x within four FP32 steps of b*S, an exact host emulation of these three roundings gives
// RN(x/S) itself (checked exhaustively: 604 million cases, no difference; 80 million random
// pairs elsewhere, S near the top of its binade included, agree too), so away from those
// neighbourhoods a quotient one step off cannot cross a boundary either; the device results are
// compared with the oracle's IEEE divisions on inputs built around the boundaries with
// full-width scales.  Scaling x and S by the same power
// of two changes none of the roundings while nothing underflows or overflows: the caller takes
// this path only for S in [2^-90, 2^90] with |x| <= 8*S, where the reciprocal, the quotient and
// the residual of any quotient >= 2^-3 stay normal, and a smaller quotient (far below the first
// boundary, 0.25) only has to keep the sign of x.
__device__ __forceinline__ float div_rn_by_recip(float x, float S, float r) {
  const float q0 = __fmul_rn(x, r);
  const float res = __fmaf_rn(-q0, S, x);
  return copysignf(__fmaf_rn(res, r, q0), x);
}

__device__ __forceinline__ void quant_block16(const float* x, float ts, uint32_t& lo, uint32_t& hi,
                                              uint32_t& sf) {
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(x[i]));
  lo = hi = 0u;
  sf = 0u;
  if (bamax == 0.0f) return;
  const float t = __fdiv_rn(__fdiv_rn(bamax, 6.0f), ts);
  sf = f32_to_e4m3(t);
  const float S = __fmul_rn(e4m3_to_f32(sf), ts);
  if (S == 0.0f) return;
  float q[16];
  if (S >= 0x1p-90f && S <= 0x1p90f && bamax <= 8.0f * S) {
    const float r = __frcp_rn(S);
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = div_rn_by_recip(x[i], S, r);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(x[i], S);
  }
  lo = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
  hi = e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
}

// The same block quantisation with reciprocal multiplies instead of divisions, for the
// intermediate h of the layer (whose codes are compared within one code step, not bit for bit):
//   sf = E4M3(max|x| * (1/6) * inv_ts); code_i = E2M1(x_i * (1 / (decode(sf) * ts))).
// It differs from quant_block16 only when a quotient lies within an ulp of a rounding boundary.
__device__ __forceinline__ void quant_block16_fast(const float* x, float ts, float inv_ts,
                                                   uint32_t& lo, uint32_t& hi, uint32_t& sf) {
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(x[i]));
  lo = hi = 0u;
  sf = 0u;
  if (bamax == 0.0f) return;
  sf = f32_to_e4m3(bamax * (1.0f / 6.0f) * inv_ts);
  const float S = e4m3_to_f32(sf) * ts;
  if (S == 0.0f) return;
  const float r = __frcp_rn(S);
  lo = e2m1x8(x[0] * r, x[1] * r, x[2] * r, x[3] * r, x[4] * r, x[5] * r, x[6] * r, x[7] * r);
  hi = e2m1x8(x[8] * r, x[9] * r, x[10] * r, x[11] * r, x[12] * r, x[13] * r, x[14] * r,
              x[15] * r);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// ---- MX formats (one E8M0 scale per 32 elements, value 2^(byte - 127)) ----
// Scale byte of a block whose largest magnitude is amax, for elements whose largest power of two
// is 2^emax (E2M1: 2, E4M3: 8): 2^(floor(log2 amax) - emax), the byte clamped to [0, 254]; 0 for
// an all-zero block.  floor(log2) is read off the exponent field (normal) or the leading bit of
// the fraction (subnormal), so it is exact.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax, int emax) {
  if (!(amax > 0.0f)) return 0u;
  const uint32_t u = __float_as_uint(amax);
  const int ef = (int)((u >> 23) & 0xFFu);
  const int fl = ef > 0 ? ef - 127 : (31 - __clz(u & 0x7FFFFFu)) - 149;
  const int b = fl - emax + 127;
  return (uint32_t)(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// 2^(byte - 127) as an FP32 value (byte 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  return b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// x / 2^(byte - 127): a multiplication by a power of two, exact unless the product underflows.
__device__ __forceinline__ float mx_unscale(float x, uint32_t b) {
  return ldexpf(x, 127 - (int)b);
}

// GEMM1's activation of one feature from its FP32 gate and up values (kAct* of internal.h; g is
// unused by the non-gated ReLU2).  Fast exponential and division: h is requantised right after
// and compared within one code step.  For a very negative argument the denominator overflows to
// infinity and the sigmoid term is a signed zero.
__device__ __forceinline__ float glu_activation(float g, float u, int act, float L, float alpha) {
  if (act == 2) return u > 0.0f ? u * u : 0.0f;   // kActRelu2
  if (act == 1 || act == 3) {                     // clamped: gate from above, up on both sides
    g = fminf(g, L);
    u = fminf(fmaxf(u, -L), L);
  }
  if (act == 3)                                   // kActSwigluOai
    return (u + 1.0f) * __fdividef(g, 1.0f + __expf(-(alpha * g)));
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// NVFP4 quantisation of one BF16 block held in registers (v0: elements 0-7, v1: elements 8-15).
__device__ __forceinline__ void quant_bf16_regs16(uint4 v0, uint4 v1, float ts, uint32_t& lo,
                                                  uint32_t& hi, uint32_t& sf) {
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
  quant_block16(f, ts, lo, hi, sf);
}

// NVFP4 quantisation of BF16 block b (elements 16b .. 16b+15 of x) with tensor scale ts.
__device__ __forceinline__ void quant_bf16_block16(const uint4* __restrict__ x, int64_t b, float ts,
                                                   uint32_t& lo, uint32_t& hi, uint32_t& sf) {
  quant_bf16_regs16(__ldg(x + 2 * b), __ldg(x + 2 * b + 1), ts, lo, hi, sf);
}

// NVFP4 encode of BF16 block b (elements 16b .. 16b+15 of x): 8 code bytes and 1 scale byte.
__device__ __forceinline__ void encode_bf16_block16(const uint4* __restrict__ x, int64_t b,
                                                    float ts, uint2* __restrict__ codes,
                                                    uint8_t* __restrict__ sf) {
  const uint4 v0 = __ldg(x + 2 * b), v1 = __ldg(x + 2 * b + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
  uint32_t lo, hi, s;
  quant_block16(f, ts, lo, hi, s);
  codes[b] = make_uint2(lo, hi);
  sf[b] = (uint8_t)s;
}

__device__ __forceinline__ uint32_t abs_bf16_max8(uint4 v) {
  uint32_t a = max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu);
  uint32_t b = max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu);
  uint32_t c = max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu);
  uint32_t d = max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu);
  return max(max(a, b), max(c, d));
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  return m;  // valid in warp 0
}



// ---------------------------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, bounded waits.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Thread-block clusters: rank of this CTA, a full cluster barrier (release / acquire, so global
// and shared writes before it are visible to every CTA of the cluster after it) and a 32-bit
// load from another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// The two halves of cluster_sync, for work that fits between them.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(const void* local_smem, uint32_t rank) {
  uint32_t ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local_smem)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}


__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// try_wait with an explicit suspend limit: a thread whose phase is not complete sleeps until the
// phase completes or kTryWaitSuspendNs pass, instead of polling at the hardware's default
// interval, so waiting warps leave the issue slots to the ones doing work.
constexpr uint32_t kTryWaitSuspendNs = 1000000u;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kTryWaitSuspendNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Counters that CTAs of one grid use to publish data to each other: a GPU-scope release add
// (after the data's stores) and a GPU-scope acquire load (before the data's loads).
__device__ __forceinline__ void red_release_add_s32(int32_t* addr, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_s32(int32_t* addr, int32_t v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t ld_acquire_s32(const int32_t* addr) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
// Orders this thread's global accesses through ordinary loads and stores with its accesses
// through the copy engine (TMA / bulk copies), in both directions.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase with the given parity; gives up after `limit_ns` nanoseconds, records
// MOE_ERR_DEVICE_TIMEOUT in the status word and returns false.  A wait that succeeds at once costs
// the poll alone; after that each poll sleeps until the phase completes or the suspend limit
// passes, and the clock is read between polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      set_status(status, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// Copies into shared memory.
// ---------------------------------------------------------------------------------------------

// 2-D tiled TMA load (box from the tensor map) completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk reduce-add of `bytes` (a multiple of 16; both addresses 16-byte aligned) FP32 values from
// shared memory into global memory, element by element, performed by the memory system; tracked
// by this thread's bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   dst),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// at most N of this thread's bulk groups still read their shared-memory source
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// at most N of this thread's bulk groups are incomplete (their global writes included)
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte cp.async with zero fill of the bytes beyond src_bytes (0 or 16).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// 4-byte cp.async with zero fill.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) wrappers.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Signals `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Copies a 32-row x 128-bit block of shared memory into tensor memory, replicated into the four
// 32-lane sub-partitions (the scale-factor copy for a 128-row block-scaled operand).
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D (+)= (A * sfA) x (B * sfB)^T with FP4 E2M1 operands and per-16 E4M3 scale factors.
__device__ __forceinline__ void tc_mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread (thread i <- lane i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading/stride byte offsets,
// descriptor version 1 at bits 46-47, layout type at bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

constexpr uint32_t kLayoutSwizzleNone = 0;
constexpr uint32_t kLayoutSwizzle128B = 2;

// Vector reduction-add of four FP32 values into global memory.
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace nvfp4moe
