// Test-only probe of the tensor-core building blocks in umma.cuh: one CTA loads
// A [M x K] and B [N x K] (bf16, row-major) into K-major SW128 shared-memory
// tiles, issues D = A B^T with tcgen05.mma, and dumps all 128 TMEM lanes x N
// columns of the fp32 accumulator so the host can check the layout.
#include <cuda_bf16.h>
#include <stdint.h>

#include "umma.cuh"

using namespace gdn::tc;

__global__ void k_umma_check(const __nv_bfloat16* A, const __nv_bfloat16* B, float* out, int M,
                             int N, int K, int ncols, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int KB = (K + 63) / 64;
  uint8_t* sA = sm;
  uint8_t* sB = sA + (size_t)M * 128 * KB;
  uint64_t* bar = (uint64_t*)(sB + (size_t)N * 128 * KB);
  uint32_t* tslot = (uint32_t*)(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < M * 64 * KB; i += blockDim.x) {
    const int r = i / (64 * KB), k = i % (64 * KB);
    *(__nv_bfloat16*)(sA + sw128_offset(r, k, M)) = k < K ? A[r * K + k] : __float2bfloat16(0.f);
  }
  for (int i = tid; i < N * 64 * KB; i += blockDim.x) {
    const int r = i / (64 * KB), k = i % (64 * KB);
    *(__nv_bfloat16*)(sB + sw128_offset(r, k, N)) = k < K ? B[r * K + k] : __float2bfloat16(0.f);
  }
  fence_async_smem();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, (uint32_t)ncols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    mma_tile(tmem, smem_u32(sA), M, smem_u32(sB), N, K, 0u);
    mma_commit(bar);
  }
  const bool ok = mbar_wait(bar, 0, 1000000000ull);
  if (!ok && lane == 0) atomicExch(status, 1);
  fence_after_sync();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) out[(32 * warp + lane) * N + c + j] = v[j];
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
}

extern "C" int umma_check(const void* A, const void* B, float* out, int M, int N, int K,
                          int* status) {
  int ncols = 32;
  while (ncols < N) ncols <<= 1;
  const int KB = (K + 63) / 64;
  const size_t smem = 1024 + (size_t)(M + N) * 128 * KB + 64;
  cudaFuncSetAttribute(k_umma_check, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_umma_check<<<1, 128, smem>>>((const __nv_bfloat16*)A, (const __nv_bfloat16*)B, out, M, N, K,
                                 ncols, status);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
}
