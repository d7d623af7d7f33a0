// Routing building blocks shared by the plan kernels and the fused small-batch prologue:
// block scan, the warp top-k of one token, its renormalised softmax weights, and the whole
// plan of a small batch inside one 1024-thread block.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

constexpr int kMaxVpl = 32;             // experts per lane: E <= 1024
constexpr int kSmallPlanThreads = 1024;

// Exclusive scan of one value per thread over the block (blockDim.x <= 1024).
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* sw, int32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sw[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t s = lane < nw ? sw[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) sw[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  total = sw[nw - 1];
  const int32_t r = (warp ? sw[warp - 1] : 0) + x - v;
  __syncthreads();
  return r;
}

// Order-preserving map of a float to an unsigned key (larger float -> larger key); -0 is folded
// into +0 so that the two compare equal, as floats do.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The variant router's expert score sqrt(softplus(x)), softplus(x) = x above 20.
__device__ __forceinline__ float sqrt_softplus(float x) {
  return sqrtf(x > 20.0f ? x : log1pf(expf(x)));
}

// Top-k of one token's logits by one warp: lane l holds experts l, l+32, ...  Each of the k
// rounds takes the warp maximum of the lanes' best keys, then the lowest expert index among the
// lanes holding it (hardware redux.sync), so ties go to the lower index.  Lane j < k ends with
// the j-th choice (my_id, my_l).  SQRTSP: the keys are sqrt(softplus(logit)) + bias[e] (bias may
// be null) and my_l is the unbiased score sqrt(softplus(logit)); otherwise keys and my_l are the
// logits.
template <int VPL, bool SQRTSP = false>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane,
                                          int& my_id, float& my_l,
                                          const float* __restrict__ bias = nullptr) {
  float v[VPL];
  uint32_t key[VPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float l = __ldg(row + e);
      if constexpr (SQRTSP) {
        v[i] = sqrt_softplus(l);
        key[i] = order_key(v[i] + (bias ? __ldg(bias + e) : 0.0f));
      } else {
        v[i] = l;
        key[i] = order_key(l);
      }
    } else {
      v[i] = 0.0f;
      key[i] = 0u;
      taken |= 1u << i;
    }
  }
  my_id = 0;
  my_l = 0.0f;
  for (int j = 0; j < k; ++j) {
    int bi = -1;
    uint32_t bk = 0u;
    float bv = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (!((taken >> i) & 1u) && (bi < 0 || key[i] > bk)) { bk = key[i]; bv = v[i]; bi = i; }
    const uint32_t lane_key = bi < 0 ? 0u : bk;
    const uint32_t mk = __reduce_max_sync(0xffffffffu, lane_key);
    const uint32_t cand = (bi >= 0 && lane_key == mk) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
    const uint32_t be = __reduce_min_sync(0xffffffffu, cand);
    const float wv = __shfl_sync(0xffffffffu, bv, (int)(be & 31u));
    if ((int)(be & 31u) == lane) taken |= 1u << (be >> 5);
    if (lane == j) { my_id = (int)be; my_l = wv; }
  }
}

// Renormalised softmax weights of the k chosen logits, summed in slot order; lanes < k write.
// SQRTSP: the chosen (unbiased) scores divided by their sum, summed in slot order.
template <bool SQRTSP = false>
__device__ __forceinline__ float topk_weight(float my_l, int k, int lane) {
  if constexpr (SQRTSP) {
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum = sum + __shfl_sync(0xffffffffu, my_l, j);
    return __fdiv_rn(my_l, sum);
  }
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum = sum + __shfl_sync(0xffffffffu, ex, j);
  return __fdiv_rn(ex, sum);
}

// Dynamic shared memory of small_plan_body for E experts.
__host__ __device__ inline size_t small_plan_smem_bytes(int E) {
  return (size_t)3 * E * sizeof(int32_t) + (size_t)kSmallPlanRows * (sizeof(int32_t) + sizeof(float)) +
         (size_t)(kSmallPlanThreads / 32) * E * sizeof(uint16_t);
}

// Place the T*k assignments of a small batch (T*k <= kSmallPlanRows) whose expert ids and router
// weights sit in s_ids / s_w and whose per-expert counts sit in s_cnt: scan the counts into
// offsets (and 128-row tile starts), then put assignment a at offsets[e] + #(earlier assignments
// to e).  Assignments are taken 1024 at a time; inside a group a warp ranks equal experts with
// match_any and each warp adds the counts of the warps before it; a per-expert cursor carries
// the counts of earlier groups.  Must be called by all kSmallPlanThreads threads of the block;
// `dyn` is the dynamic shared memory laid out as in small_plan_body.  Every global output may be
// null (nothing written).
__device__ __forceinline__ void small_place(int T, int E, int k, int shared_rows,
                                            int32_t* __restrict__ counts,
                                            int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ tile_start,
                                            int32_t* __restrict__ perm_src,
                                            float* __restrict__ perm_w, int32_t* __restrict__ inv,
                                            uint8_t* dyn, int32_t* __restrict__ perm_seg) {
  int32_t* s_cnt = reinterpret_cast<int32_t*>(dyn);
  int32_t* s_off = s_cnt + E;
  int32_t* s_cur = s_off + E;
  int32_t* s_ids = s_cur + E;
  float* s_w = reinterpret_cast<float*>(s_ids + kSmallPlanRows);
  uint16_t* s_wcnt = reinterpret_cast<uint16_t*>(s_w + kSmallPlanRows);
  __shared__ int32_t sw[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kSmallPlanThreads / 32;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cur[e] = 0;
  const int e = threadIdx.x;
  const int32_t cnt = e < E ? s_cnt[e] : 0;
  int32_t total, ttotal;
  const int32_t off = block_exclusive_scan(cnt, sw, total);
  const int32_t toff = block_exclusive_scan((cnt + kBM - 1) / kBM, sw, ttotal);
  if (e < E) {
    s_off[e] = off;
    if (counts) counts[e] = cnt;
    if (offsets) offsets[e] = off;
    if (tile_start) tile_start[e] = toff;
  }
  if (threadIdx.x == 0) {
    if (offsets) offsets[E] = total;
    if (offsets && shared_rows > 0) offsets[E + 1] = total + shared_rows;
    if (tile_start) {
      tile_start[E] = ttotal;
      if (shared_rows > 0) tile_start[E + 1] = ttotal + (shared_rows + kBM - 1) / kBM;
    }
  }
  const int R = T * k;
  const uint32_t lt = (1u << lane) - 1u;
  for (int a0 = 0; a0 < R; a0 += kSmallPlanThreads) {
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) s_wcnt[i] = 0;
    __syncthreads();
    const int a = a0 + threadIdx.x;
    const bool valid = a < R;
    const int ea = valid ? s_ids[a] : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, ea);
    if (valid && (peers & lt) == 0) s_wcnt[warp * E + ea] = (uint16_t)__popc(peers);
    __syncthreads();
    if (valid) {
      int rank = __popc(peers & lt) + s_cur[ea];
      for (int v = 0; v < warp; ++v) rank += s_wcnt[v * E + ea];
      const int p = s_off[ea] + rank;
      if (perm_src) perm_src[p] = a / k;
      if (perm_w) perm_w[p] = s_w[a];
      if (perm_seg) perm_seg[p] = ea;
      if (inv) inv[a] = p;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      int col = 0;
      for (int v = 0; v < nw; ++v) col += s_wcnt[v * E + x];
      s_cur[x] += col;
    }
    __syncthreads();
  }
  for (int t = threadIdx.x; t < shared_rows && perm_src; t += blockDim.x) {
    perm_src[R + t] = t;
    if (perm_w) perm_w[R + t] = 1.0f;
    if (perm_seg) perm_seg[R + t] = E;
  }
}

// Route T tokens (T*k <= kSmallPlanRows) inside one block, count per expert, then place (above).
template <int VPL, bool SQRTSP>
__device__ __forceinline__ void small_plan_body(
    const float* __restrict__ logits, int T, int E, int k, int shared_rows,
    int32_t* __restrict__ ids, float* __restrict__ wout, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_start,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w, int32_t* __restrict__ inv,
    uint8_t* dyn, int32_t* __restrict__ perm_seg = nullptr,
    const float* __restrict__ bias = nullptr) {
  int32_t* s_cnt = reinterpret_cast<int32_t*>(dyn);
  int32_t* s_ids = s_cnt + 3 * E;
  float* s_w = reinterpret_cast<float*>(s_ids + kSmallPlanRows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kSmallPlanThreads / 32;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int t = warp; t < T; t += nw) {
    int my_id;
    float my_l;
    warp_topk<VPL, SQRTSP>(logits + (int64_t)t * E, E, k, lane, my_id, my_l, bias);
    const float w = topk_weight<SQRTSP>(my_l, k, lane);
    if (lane < k) {
      ids[(int64_t)t * k + lane] = my_id;
      wout[(int64_t)t * k + lane] = w;
      s_ids[t * k + lane] = my_id;
      s_w[t * k + lane] = w;
      atomicAdd(&s_cnt[my_id], 1);
    }
  }
  __syncthreads();
  small_place(T, E, k, shared_rows, counts, offsets, tile_start, perm_src, perm_w, inv, dyn,
              perm_seg);
}

}  // namespace nvfp4moe
