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
#include "route.cuh"

namespace nvfp4moe {

namespace {

constexpr int kRouterWarps = 8;

// One warp per token; the per-chunk expert histogram (chunk = tpc tokens) is accumulated with
// global atomics into `hist`, which the caller zeroes first.
template <int VPL, bool SQRTSP>
__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(
    const float* __restrict__ logits, int T, int E, int k, int tpc, int32_t* __restrict__ ids,
    float* __restrict__ wout, int32_t* __restrict__ hist, const float* __restrict__ bias) {
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouterWarps + warp;
  if (t >= T) return;
  int my_id;
  float my_l;
  warp_topk<VPL, SQRTSP>(logits + (int64_t)t * E, E, k, lane, my_id, my_l, bias);
  const float w = topk_weight<SQRTSP>(my_l, k, lane);
  if (lane < k) {
    ids[(int64_t)t * k + lane] = my_id;
    wout[(int64_t)t * k + lane] = w;
    atomicAdd(hist + (int64_t)(t / tpc) * E + my_id, 1);
  }
}

template <int VPL, bool SQRTSP>
__global__ void __launch_bounds__(kSmallPlanThreads) plan_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int shared_rows,
    int32_t* __restrict__ ids, float* __restrict__ wout, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_start,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w, int32_t* __restrict__ inv,
    int32_t* __restrict__ perm_seg, const float* __restrict__ bias) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  griddep_wait();
  griddep_launch();
  small_plan_body<VPL, SQRTSP>(logits, T, E, k, shared_rows, ids, wout, counts, offsets,
                               tile_start, perm_src, perm_w, inv, s_dyn, perm_seg, bias);
}

// Per-chunk bases and per-expert offsets from the chunk histograms, spread over blocks of 32
// experts: lane l of every warp owns expert 32*block + l (so each chunk row is read coalesced),
// warp w sums a contiguous range of chunks, a scan over the 32 warp sums gives each range its
// start, and the range is written out as running sums.  The block that finishes last (atomic
// count, reset to 0 for the next call) scans the per-expert totals into offsets and 128-row tile
// starts.  scratch[0] is that count, scratch[1..E] the totals.
__global__ void __launch_bounds__(1024) plan_scan_kernel(const int32_t* __restrict__ hist,
                                                        int nchunks, int E, int shared_rows,
                                                        int32_t* __restrict__ base,
                                                        int32_t* __restrict__ counts,
                                                        int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ tile_start,
                                                        int32_t* __restrict__ scratch) {
  __shared__ int32_t s_part[32][33];
  __shared__ int32_t sw[32];
  __shared__ int s_last;
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  const int cpw = (nchunks + 31) / 32;
  const int c0 = min(nchunks, warp * cpw), c1 = min(nchunks, c0 + cpw);
  int32_t sum = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) sum += __ldcg(hist + (int64_t)c * E + e);
  s_part[warp][lane] = sum;
  __syncthreads();
  int32_t run = 0;
  for (int v = 0; v < warp; ++v) run += s_part[v][lane];
  if (e < E) {
    if (warp == 31) scratch[1 + e] = run + sum;   // the expert's total
    for (int c = c0; c < c1; ++c) {
      const int32_t h = __ldcg(hist + (int64_t)c * E + e);
      base[(int64_t)c * E + e] = run;
      run += h;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(scratch, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int t = threadIdx.x;
  const int32_t cnt = t < E ? __ldcg(scratch + 1 + t) : 0;
  int32_t total;
  const int32_t off = block_exclusive_scan(cnt, sw, total);
  const int32_t ntile = (cnt + kBM - 1) / kBM;
  int32_t ttotal;
  const int32_t toff = block_exclusive_scan(ntile, sw, ttotal);
  if (t < E) {
    if (counts) counts[t] = cnt;
    offsets[t] = off;
    if (tile_start) tile_start[t] = toff;
  }
  if (t == 0) {
    offsets[E] = total;
    const int32_t shared_tiles = (shared_rows + kBM - 1) / kBM;
    if (shared_rows > 0) offsets[E + 1] = total + shared_rows;
    if (tile_start) {
      tile_start[E] = ttotal;
      if (shared_rows > 0) tile_start[E + 1] = ttotal + shared_tiles;
    }
    scratch[0] = 0;
  }
}

// One block per token chunk: stable rank of every assignment among the chunk's assignments to
// the same expert, then p = offsets[e] + base[chunk][e] + rank.
__global__ void __launch_bounds__(1024) plan_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int E, int k, int tpc,
    int shared_rows, const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w, int32_t* __restrict__ inv,
    int32_t* __restrict__ perm_seg) {
  extern __shared__ int32_t s_wcnt[];  // [nwarps][E]
  griddep_wait();
  griddep_launch();
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
    if (perm_seg) perm_seg[p] = e;
    inv[a] = p;
  }
  if (shared_rows > 0) {  // the shared expert's rows: token t at row R + t, weight 1
    const int t0 = blockIdx.x * tpc;
    for (int t = t0 + threadIdx.x; t < min(T, t0 + tpc); t += blockDim.x) {
      perm_src[R + t] = t;
      if (perm_w) perm_w[R + t] = 1.0f;
      if (perm_seg) perm_seg[R + t] = E;
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
  const int tpc = plan_tokens_per_chunk(a.k);
  const int nchunks = (a.T + tpc - 1) / tpc;
  const int vpl = (a.E + 31) / 32;
  if ((int64_t)a.T * a.k <= kSmallPlanRows) {
    const size_t smem = small_plan_smem_bytes(a.E);
#define NVFP4MOE_SMALL2(V, SP)                                                                  \
  do {                                                                                          \
    if (smem > 48 * 1024)                                                                       \
      cudaFuncSetAttribute(plan_small_kernel<V, SP>,                                            \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);             \
    cudaError_t le = launch_pdl(plan_small_kernel<V, SP>, dim3(1), dim3(kSmallPlanThreads), smem, \
        s, a.logits, a.T, a.E, a.k, a.shared_rows, a.ids, a.w, a.counts, a.offsets,             \
        a.tile_start, a.perm_src, a.perm_w, a.inv, a.perm_seg, a.bias);                         \
    if (le != cudaSuccess) return le;                                                           \
  } while (0)
#define NVFP4MOE_SMALL(V)                                                                       \
  do {                                                                                          \
    if (a.sqrtsp) NVFP4MOE_SMALL2(V, true);                                                     \
    else NVFP4MOE_SMALL2(V, false);                                                             \
  } while (0)
    if (vpl <= 1) NVFP4MOE_SMALL(1);
    else if (vpl <= 2) NVFP4MOE_SMALL(2);
    else if (vpl <= 4) NVFP4MOE_SMALL(4);
    else if (vpl <= 8) NVFP4MOE_SMALL(8);
    else if (vpl <= 16) NVFP4MOE_SMALL(16);
    else NVFP4MOE_SMALL(kMaxVpl);
#undef NVFP4MOE_SMALL
#undef NVFP4MOE_SMALL2
    return cudaGetLastError();
  }
  // the histograms and the scan's block count (scratch after them) start at zero
  cudaError_t err = cudaMemsetAsync(a.hist, 0, sizeof(int32_t) * ((size_t)nchunks * a.E + 1), s);
  if (err != cudaSuccess) return err;
  const int rblocks = (a.T + kRouterWarps - 1) / kRouterWarps;
#define NVFP4MOE_ROUTER(V)                                                                 \
  err = a.sqrtsp                                                                            \
            ? launch_pdl(router_kernel<V, true>, dim3(rblocks), dim3(kRouterWarps * 32), 0, s, \
                         a.logits, a.T, a.E, a.k, tpc, a.ids, a.w, a.hist, a.bias)          \
            : launch_pdl(router_kernel<V, false>, dim3(rblocks), dim3(kRouterWarps * 32), 0, s, \
                         a.logits, a.T, a.E, a.k, tpc, a.ids, a.w, a.hist, a.bias)
  if (vpl <= 1) NVFP4MOE_ROUTER(1);
  else if (vpl <= 2) NVFP4MOE_ROUTER(2);
  else if (vpl <= 4) NVFP4MOE_ROUTER(4);
  else if (vpl <= 8) NVFP4MOE_ROUTER(8);
  else if (vpl <= 16) NVFP4MOE_ROUTER(16);
  else NVFP4MOE_ROUTER(kMaxVpl);
#undef NVFP4MOE_ROUTER
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = launch_pdl(plan_scan_kernel, dim3((a.E + 31) / 32), dim3(1024), 0, s,
                   (const int32_t*)a.hist, nchunks, a.E, a.shared_rows, a.base, a.counts,
                   a.offsets, a.tile_start, a.hist + (size_t)nchunks * a.E);
  if (err != cudaSuccess) return err;
  const int threads = ((tpc * a.k + 31) / 32) * 32;
  const size_t sc_smem = sizeof(int32_t) * (threads / 32) * a.E;
  if (sc_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(plan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sc_smem);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(plan_scatter_kernel, dim3(nchunks), dim3(threads), sc_smem, s,
                    (const int32_t*)a.ids, (const float*)a.w, a.T, a.E, a.k, tpc, a.shared_rows,
                    (const int32_t*)a.base, (const int32_t*)a.offsets, a.perm_src, a.perm_w, a.inv,
                    a.perm_seg);
}

}  // namespace nvfp4moe
