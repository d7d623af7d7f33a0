// Pure read bandwidth of this GPU by three load paths, one CTA per SM, each CTA streaming its own
// contiguous 4 MiB: (A) cp.async.bulk copies into an mbarrier ring, (B) per-thread 16-byte
// cp.async with a 16-deep wait_group pipeline, (C) 16-byte ld.global.nc into registers, and
// (A) with half of each CTA range read by (B) alongside.  Every CTA reads only inside its own
// range; every wait is bounded.  Build and run (from the repository root):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o /tmp/read_bw nvfp4_mixture_experts_softmax_gb300/probes/read_bw.cu && /tmp/read_bw
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t par) {
  uint32_t ok;
  asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0,1,0,p;\n}" : "=r"(ok) : "r"(bar), "r"(par) : "memory");
  return ok;
}
__device__ __forceinline__ uint64_t gt() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ bool wait_b(uint32_t bar, uint32_t par, int* err) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (try_wait(bar, par)) return true;
    if ((i & 1023) == 1023) { uint64_t n = gt(); if (!t0) t0 = n; else if (n - t0 > 1000000000ull) { atomicExch(err, 1); return false; } }
  }
}

// (A) bulk ring by thread 0 (consumer thread 32 releases at once); optional (D): warps 2.. stream
// a disjoint second half of the CTA's range with cp.async
template <bool kMixed>
__global__ void __launch_bounds__(256, 1) probe_bulk(const uint8_t* src, size_t per_cta, int stage, int nst,
                                                     int* err, unsigned long long* sink) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* full = (uint64_t*)(sm + (size_t)nst * stage);
  uint64_t* empty = full + nst;
  uint8_t* cpa = (uint8_t*)(empty + nst) + 64;   // cp.async scratch: 6 warps x 32 thr x 16 deep x 16 B = 48 KB
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su32(full + s)));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su32(empty + s)));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const size_t bulk_bytes = kMixed ? per_cta / 2 : per_cta;
  const uint8_t* base = src + (size_t)blockIdx.x * per_cta;
  const int n = (int)(bulk_bytes / stage);
  if (threadIdx.x == 0) {
    int s = 0; uint32_t ph = 0;
    for (int i = 0; i < n; ++i) {
      if (!wait_b(su32(empty + s), ph ^ 1, err)) break;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(su32(full + s)), "r"(stage) : "memory");
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   :: "r"(su32(sm + (size_t)s * stage)), "l"(base + (size_t)i * stage), "r"(stage), "r"(su32(full + s)) : "memory");
      if (++s == nst) { s = 0; ph ^= 1; }
    }
    for (int i = 0; i < nst; ++i) { if (!wait_b(su32(empty + s), ph ^ 1, err)) break; if (++s == nst) { s = 0; ph ^= 1; } }
  } else if (threadIdx.x == 32) {
    int s = 0; uint32_t ph = 0; unsigned long long acc = 0;
    for (int i = 0; i < n; ++i) {
      if (!wait_b(su32(full + s), ph, err)) break;
      acc += sm[(size_t)s * stage + (i & 1023)];
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(su32(empty + s)) : "memory");
      if (++s == nst) { s = 0; ph ^= 1; }
    }
    if (acc == 0x123456789ull) *sink = acc;
  } else if (kMixed && threadIdx.x >= 64) {
    // 192 threads, 16 B each per round, 16 rounds deep
    const int t = threadIdx.x - 64;
    const uint8_t* b2 = base + bulk_bytes;
    const size_t rounds = (per_cta - bulk_bytes) / (192 * 16);
    const uint32_t my = su32(cpa + (size_t)t * 16 * 16);
    for (size_t r = 0; r < rounds; ++r) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(my + (uint32_t)(r & 15) * 16), "l"(b2 + (r * 192 + t) * 16) : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 15;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  __syncthreads();
}

// (B) cp.async only: every thread, `depth` deep
__global__ void __launch_bounds__(512, 1) probe_cpasync(const uint8_t* src, size_t per_cta, unsigned long long* sink) {
  extern __shared__ __align__(1024) uint8_t sm[];
  const int nt = blockDim.x, t = threadIdx.x;
  const uint8_t* base = src + (size_t)blockIdx.x * per_cta;
  const size_t rounds = per_cta / ((size_t)nt * 16);
  const uint32_t my = su32(sm + (size_t)t * 16 * 16);
  for (size_t r = 0; r < rounds; ++r) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(my + (uint32_t)(r & 15) * 16), "l"(base + (r * nt + t) * 16) : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 15;" ::: "memory");
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  if (sm[t] == 0x7f && t == 1000000) *sink = 1;
}

// (C) ld.global.nc.v4 into registers, 8 loads in flight per thread
__global__ void __launch_bounds__(1024, 1) probe_ldg(const uint8_t* src, size_t per_cta, unsigned long long* sink) {
  const int nt = blockDim.x, t = threadIdx.x;
  const uint4* base = reinterpret_cast<const uint4*>(src + (size_t)blockIdx.x * per_cta);
  const size_t n = per_cta / 16;
  uint32_t acc = 0;
  for (size_t i = t; i + 7 * (size_t)nt < n; i += 8 * (size_t)nt) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldg(base + i + (size_t)u * nt);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].w;
  }
  if (acc == 0x12345678u) *sink = acc;
}

int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t per_cta = 4u << 20;
  const size_t total = per_cta * sms;
  uint8_t* buf; int* err; unsigned long long* sink; uint8_t* flush;
  if (cudaMalloc(&buf, total) || cudaMalloc(&err, 4) || cudaMalloc(&sink, 8) || cudaMalloc(&flush, 512u << 20)) { printf("alloc fail\n"); return 1; }
  cudaMemset(buf, 1, total); cudaMemset(err, 0, 4);
  cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
  auto timeit = [&](const char* name, auto launch) {
    float best = 1e9;
    for (int rep = 0; rep < 5; ++rep) {
      cudaMemset(flush, rep, 512u << 20);
      cudaEventRecord(a); launch(); cudaEventRecord(b); cudaEventSynchronize(b);
      float ms; cudaEventElapsedTime(&ms, a, b); if (ms < best) best = ms;
    }
    int h = 0; cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
    printf("%-34s %8.1f GB/s (%.1f us) err=%d cuda=%s\n", name, (double)total / (best * 1e-3) / 1e9, best * 1e3, h,
           cudaGetErrorString(cudaGetLastError()));
  };
  const int stage = 18432;
  for (int nst : {4, 8}) {
    size_t smem = (size_t)nst * stage + 1024 + 64 + 49152;
    cudaFuncSetAttribute(probe_bulk<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(probe_bulk<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    char nm[64];
    snprintf(nm, 64, "bulk nst=%d", nst);
    timeit(nm, [&] { probe_bulk<false><<<sms, 256, smem>>>(buf, per_cta, stage, nst, err, sink); });
    snprintf(nm, 64, "bulk+cp.async nst=%d", nst);
    timeit(nm, [&] { probe_bulk<true><<<sms, 256, smem>>>(buf, per_cta, stage, nst, err, sink); });
  }
  for (int thr : {256, 512}) {
    size_t smem = (size_t)thr * 256;
    cudaFuncSetAttribute(probe_cpasync, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    char nm[64]; snprintf(nm, 64, "cp.async threads=%d depth=16", thr);
    timeit(nm, [&] { probe_cpasync<<<sms, thr, smem>>>(buf, per_cta, sink); });
  }
  for (int thr : {256, 512, 1024}) {
    char nm[64]; snprintf(nm, 64, "ldg.v4 threads=%d x8", thr);
    timeit(nm, [&] { probe_ldg<<<sms, thr>>>(buf, per_cta, sink); });
  }
  return 0;
}
