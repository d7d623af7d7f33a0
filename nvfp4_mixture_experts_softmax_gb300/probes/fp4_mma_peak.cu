// Dense FP4 tensor-core rate of this GPU: tcgen05.mma kind::mxf4nvf4 (E2M1 operands, UE4M3 scale
// per 16 elements, K = 64 per instruction) issued back to back by one thread per CTA on
// shared-memory operands (no global traffic), one CTA per SM, for M = 128 and N in {64, 128, 256}.
// Build and run (from the repository root):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -Iinclude \
//        -o /tmp/fp4_mma_peak nvfp4_mixture_experts_softmax_gb300/probes/fp4_mma_peak.cu && /tmp/fp4_mma_peak
// Every wait is bounded (status word set on timeout).
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "../csrc/common.cuh"

using namespace nvfp4moe;

__global__ void __launch_bounds__(128, 1) fp4_probe(int N, int iters, int32_t* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  // A: 128 rows x 128 B; B: 256 rows x 128 B; SF: 2 x 2 KB; bars
  uint8_t* A = sm;
  uint8_t* B = sm + 16384;
  uint8_t* SF = B + 32768;
  uint64_t* bar = reinterpret_cast<uint64_t*>(SF + 4096);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  for (int i = threadIdx.x; i < (16384 + 32768 + 4096) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x22222222u;   // E2M1 1.0 codes; scale bytes 0x22
  if (threadIdx.x < 32) { tmem_alloc(smem_u32(slot), 512); tmem_relinquish(); }
  if (threadIdx.x == 0) { mbar_init(smem_u32(bar), 1); fence_barrier_init(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint32_t sfa = tm + 256, sfb = tm + 256 + 32;   // B: 8 columns per K step (N up to 256)
    for (int kk = 0; kk < 4; ++kk) {
      tc_cp_32x128b_warpx4(sfa + kk * 4, smem_desc(smem_u32(SF) + kk * 512, 0, 128, kLayoutSwizzleNone));
      tc_cp_32x128b_warpx4(sfb + kk * 8, smem_desc(smem_u32(SF + 2048) + kk * 512, 0, 128, kLayoutSwizzleNone));
      tc_cp_32x128b_warpx4(sfb + kk * 8 + 4, smem_desc(smem_u32(SF + 2048) + kk * 512, 0, 128, kLayoutSwizzleNone));
    }
    const uint64_t ad = smem_desc(smem_u32(A), 16, 1024, kLayoutSwizzle128B);
    const uint64_t bd = smem_desc(smem_u32(B), 16, 1024, kLayoutSwizzle128B);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_mxf4nvf4(tm, ad + kk * 2, bd + kk * 2, idesc, sfa + kk * 4, sfb + kk * 8, (it | kk) != 0);
    }
    tc_commit(smem_u32(bar));
    mbar_wait_bounded(smem_u32(bar), 0u, 4000000000ull, status);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  int32_t* st; cudaMalloc(&st, 4); cudaMemset(st, 0, 4);
  const size_t smem = 1024 + 16384 + 32768 + 4096 + 64;
  cudaFuncSetAttribute(fp4_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
  const int iters = 20000;
  for (int N : {64, 128, 256}) {
    float best = 1e9;
    for (int rep = 0; rep < 4; ++rep) {
      cudaEventRecord(a);
      fp4_probe<<<sms, 128, smem>>>(N, iters, st);
      cudaEventRecord(b); cudaEventSynchronize(b);
      float ms; cudaEventElapsedTime(&ms, a, b); if (ms < best) best = ms;
    }
    int h = 0; cudaMemcpy(&h, st, 4, cudaMemcpyDeviceToHost);
    const double flop = 2.0 * 128 * N * 256.0 * iters * sms;
    printf("M=128 N=%3d K=64x4 per iter: %8.1f TFLOP/s  (%.3f ms, %.1f cycles/MMA at 2.07 GHz) status=%d cuda=%s\n",
           N, flop / (best * 1e-3) / 1e12, best, best * 1e-3 * 2.07e9 / (iters * 4.0), h,
           cudaGetErrorString(cudaGetLastError()));
  }
  return 0;
}
