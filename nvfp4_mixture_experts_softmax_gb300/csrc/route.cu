// Router top-k and the token -> expert plan (histogram, scan, stable scatter), all on the device.
//
// Router: one warp per token ("vllm.cpp docs/STATUS.md", row "DeepSeek-V4-Flash decode ds4-gap -
// Lever 3 (route -> warp-topk)": experts spread over the lanes, per-lane arg-max, warp
// reduction, mask and repeat; here the reduction is two redux.sync instructions per round on an
// order-preserving integer key).  Selection is on the raw logits under the strict order (value
// descending, lower index on ties), which softmax preserves; the weights are
// w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0), summed in slot order (softmax restricted to
// the chosen k and renormalised).
//
// Plan: counts and offsets are built without any host read ("nvfp4-megamoe-kernel compare
// pre-b1...master", "CATEGORY 3: Data-dependent control flow": device scatter into a preallocated
// buffer instead of bincount).  Rows of one expert are ordered by ascending assignment index
// t*k + j, so the permutation has exactly one correct value.  Small batches (T*k <= 2048) run
// the whole plan in one block; larger ones count assignments per chunk of tokens, scan the
// counts into per-(chunk, expert) bases, and rank assignments inside a chunk with warp match +
// per-warp counts.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

constexpr int kRouterWarps = 8;
constexpr int kMaxVpl = 32;  // experts per lane: E <= 1024

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

// Top-k of one token's logits by one warp: lane l holds experts l, l+32, ...  Each of the k
// rounds takes the warp maximum of the lanes' best keys, then the lowest expert index among the
// lanes holding it (hardware redux.sync), so ties go to the lower index.  Lane j < k ends with
// the j-th choice (my_id, my_l).
template <int VPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane,
                                          int& my_id, float& my_l) {
  float v[VPL];
  uint32_t key[VPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      v[i] = __ldg(row + e);
      key[i] = order_key(v[i]);
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
__device__ __forceinline__ float topk_weight(float my_l, int k, int lane) {
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum = sum + __shfl_sync(0xffffffffu, ex, j);
  return __fdiv_rn(ex, sum);
}

// One warp per token; the per-chunk expert histogram (chunk = tpc tokens) is accumulated with
// global atomics into `hist`, which the caller zeroes first.
template <int VPL>
__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(
    const float* __restrict__ logits, int T, int E, int k, int tpc, int32_t* __restrict__ ids,
    float* __restrict__ wout, int32_t* __restrict__ hist) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouterWarps + warp;
  if (t >= T) return;
  int my_id;
  float my_l;
  warp_topk<VPL>(logits + (int64_t)t * E, E, k, lane, my_id, my_l);
  const float w = topk_weight(my_l, k, lane);
  if (lane < k) {
    ids[(int64_t)t * k + lane] = my_id;
    wout[(int64_t)t * k + lane] = w;
    atomicAdd(hist + (int64_t)(t / tpc) * E + my_id, 1);
  }
}

// The whole plan in one block for small batches (T*k <= kSmallPlanRows): route, count, scan,
// and place every assignment at offsets[e] + #(earlier assignments to e).
constexpr int kSmallPlanRows = 2048;
constexpr int kSmallPlanThreads = 1024;

template <int VPL>
__global__ void __launch_bounds__(kSmallPlanThreads) plan_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int shared_rows,
    int32_t* __restrict__ ids, float* __restrict__ wout, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_start,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w, int32_t* __restrict__ inv) {
  __shared__ int32_t s_cnt[1024];
  __shared__ int32_t s_off[1024];
  __shared__ int32_t s_ids[kSmallPlanRows];
  __shared__ float s_w[kSmallPlanRows];
  __shared__ int32_t sw[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int t = warp; t < T; t += kSmallPlanThreads / 32) {
    int my_id;
    float my_l;
    warp_topk<VPL>(logits + (int64_t)t * E, E, k, lane, my_id, my_l);
    const float w = topk_weight(my_l, k, lane);
    if (lane < k) {
      ids[(int64_t)t * k + lane] = my_id;
      wout[(int64_t)t * k + lane] = w;
      s_ids[t * k + lane] = my_id;
      s_w[t * k + lane] = w;
      atomicAdd(&s_cnt[my_id], 1);
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int32_t cnt = e < E ? s_cnt[e] : 0;
  int32_t total, ttotal;
  const int32_t off = block_exclusive_scan(cnt, sw, total);
  const int32_t toff = block_exclusive_scan((cnt + kBM - 1) / kBM, sw, ttotal);
  if (e < E) {
    s_off[e] = off;
    if (counts) counts[e] = cnt;
    offsets[e] = off;
    if (tile_start) tile_start[e] = toff;
  }
  if (threadIdx.x == 0) {
    offsets[E] = total;
    if (shared_rows > 0) offsets[E + 1] = total + shared_rows;
    if (tile_start) {
      tile_start[E] = ttotal;
      if (shared_rows > 0) tile_start[E + 1] = ttotal + (shared_rows + kBM - 1) / kBM;
    }
  }
  __syncthreads();
  const int R = T * k;
  for (int a = threadIdx.x; a < R; a += blockDim.x) {
    const int ea = s_ids[a];
    int rank = 0;
    for (int b = 0; b < a; ++b) rank += (s_ids[b] == ea);
    const int p = s_off[ea] + rank;
    perm_src[p] = a / k;
    if (perm_w) perm_w[p] = s_w[a];
    inv[a] = p;
  }
  for (int t = threadIdx.x; t < shared_rows; t += blockDim.x) {
    perm_src[R + t] = t;
    if (perm_w) perm_w[R + t] = 1.0f;
  }
}

// One block of 1024 threads: per-expert exclusive scan over chunks (base), counts, segment
// offsets and the prefix of 128-row tiles per segment.  Segment E (when shared_rows > 0) is the
// shared expert: shared_rows rows starting at T*k.
constexpr int kScanRows = 16;

__global__ void __launch_bounds__(1024) plan_scan_kernel(const int32_t* __restrict__ hist,
                                                        int nchunks, int E, int shared_rows,
                                                        int32_t* __restrict__ base,
                                                        int32_t* __restrict__ counts,
                                                        int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ tile_start) {
  extern __shared__ int32_t s_tile[];  // [kScanRows][E]
  __shared__ int32_t sw[32];
  const int e = threadIdx.x;
  int32_t run = 0;
  for (int c0 = 0; c0 < nchunks; c0 += kScanRows) {
    const int rows = min(kScanRows, nchunks - c0);
    for (int i = threadIdx.x; i < rows * E; i += blockDim.x) s_tile[i] = hist[(int64_t)c0 * E + i];
    __syncthreads();
    if (e < E)
      for (int r = 0; r < rows; ++r) {
        const int32_t v = s_tile[r * E + e];
        s_tile[r * E + e] = run;
        run += v;
      }
    __syncthreads();
    for (int i = threadIdx.x; i < rows * E; i += blockDim.x) base[(int64_t)c0 * E + i] = s_tile[i];
    __syncthreads();
  }
  const int32_t cnt = e < E ? run : 0;
  int32_t total;
  const int32_t off = block_exclusive_scan(cnt, sw, total);
  const int32_t ntile = (cnt + kBM - 1) / kBM;
  int32_t ttotal;
  const int32_t toff = block_exclusive_scan(ntile, sw, ttotal);
  if (e < E) {
    if (counts) counts[e] = cnt;
    offsets[e] = off;
    if (tile_start) tile_start[e] = toff;
  }
  if (threadIdx.x == 0) {
    offsets[E] = total;
    const int32_t shared_tiles = (shared_rows + kBM - 1) / kBM;
    if (shared_rows > 0) offsets[E + 1] = total + shared_rows;
    if (tile_start) {
      tile_start[E] = ttotal;
      if (shared_rows > 0) tile_start[E + 1] = ttotal + shared_tiles;
    }
  }
}

// One block per token chunk: stable rank of every assignment among the chunk's assignments to
// the same expert, then p = offsets[e] + base[chunk][e] + rank.
__global__ void __launch_bounds__(1024) plan_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int E, int k, int tpc,
    int shared_rows, const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w, int32_t* __restrict__ inv) {
  extern __shared__ int32_t s_wcnt[];  // [nwarps][E]
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) s_wcnt[i] = 0;
  __syncthreads();
  const int64_t R = (int64_t)T * k;
  const int64_t a0 = (int64_t)blockIdx.x * tpc * k;
  const int64_t a = a0 + threadIdx.x;
  const bool valid = threadIdx.x < tpc * k && a < R;
  const int e = valid ? ids[a] : -1 - lane;  // invalid lanes form singleton groups
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const uint32_t lt = (1u << lane) - 1u;
  const int rank_w = __popc(peers & lt);
  if (valid && (peers & lt) == 0) s_wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  if (valid) {
    int rank = rank_w;
    for (int v = 0; v < warp; ++v) rank += s_wcnt[v * E + e];
    const int32_t p = offsets[e] + base[(int64_t)blockIdx.x * E + e] + rank;
    perm_src[p] = (int32_t)(a / k);
    if (perm_w) perm_w[p] = w[a];
    inv[a] = p;
  }
  if (shared_rows > 0) {  // the shared expert's rows: token t at row R + t, weight 1
    const int t0 = blockIdx.x * tpc;
    for (int t = t0 + threadIdx.x; t < min(T, t0 + tpc); t += blockDim.x) {
      perm_src[R + t] = t;
      if (perm_w) perm_w[R + t] = 1.0f;
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
  const int tpc = plan_tokens_per_chunk(a.k);
  const int nchunks = (a.T + tpc - 1) / tpc;
  const int vpl = (a.E + 31) / 32;
  if ((int64_t)a.T * a.k <= kSmallPlanRows) {
#define NVFP4MOE_SMALL(V)                                                                     \
  plan_small_kernel<V><<<1, kSmallPlanThreads, 0, s>>>(a.logits, a.T, a.E, a.k, a.shared_rows, \
                                                       a.ids, a.w, a.counts, a.offsets,        \
                                                       a.tile_start, a.perm_src, a.perm_w, a.inv)
    if (vpl <= 1) NVFP4MOE_SMALL(1);
    else if (vpl <= 2) NVFP4MOE_SMALL(2);
    else if (vpl <= 4) NVFP4MOE_SMALL(4);
    else if (vpl <= 8) NVFP4MOE_SMALL(8);
    else if (vpl <= 16) NVFP4MOE_SMALL(16);
    else NVFP4MOE_SMALL(kMaxVpl);
#undef NVFP4MOE_SMALL
    return cudaGetLastError();
  }
  cudaError_t err = cudaMemsetAsync(a.hist, 0, sizeof(int32_t) * (size_t)nchunks * a.E, s);
  if (err != cudaSuccess) return err;
  const int rblocks = (a.T + kRouterWarps - 1) / kRouterWarps;
#define NVFP4MOE_ROUTER(V)                                                                 \
  router_kernel<V><<<rblocks, kRouterWarps * 32, 0, s>>>(a.logits, a.T, a.E, a.k, tpc, a.ids, \
                                                        a.w, a.hist)
  if (vpl <= 1) NVFP4MOE_ROUTER(1);
  else if (vpl <= 2) NVFP4MOE_ROUTER(2);
  else if (vpl <= 4) NVFP4MOE_ROUTER(4);
  else if (vpl <= 8) NVFP4MOE_ROUTER(8);
  else if (vpl <= 16) NVFP4MOE_ROUTER(16);
  else NVFP4MOE_ROUTER(kMaxVpl);
#undef NVFP4MOE_ROUTER
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t scan_smem = sizeof(int32_t) * kScanRows * a.E;
  if (scan_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(plan_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)scan_smem);
    if (err != cudaSuccess) return err;
  }
  plan_scan_kernel<<<1, 1024, scan_smem, s>>>(a.hist, nchunks, a.E, a.shared_rows, a.base,
                                              a.counts, a.offsets, a.tile_start);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int threads = ((tpc * a.k + 31) / 32) * 32;
  const size_t sc_smem = sizeof(int32_t) * (threads / 32) * a.E;
  if (sc_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(plan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sc_smem);
    if (err != cudaSuccess) return err;
  }
  plan_scatter_kernel<<<nchunks, threads, sc_smem, s>>>(a.ids, a.w, a.T, a.E, a.k, tpc,
                                                        a.shared_rows, a.base, a.offsets,
                                                        a.perm_src, a.perm_w, a.inv);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
