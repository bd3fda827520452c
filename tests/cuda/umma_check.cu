// Test-only probe of the tensor-core building blocks in umma.cuh: one CTA loads
// A [M x K] and B [N x K] (bf16, row-major) into SW128 shared-memory tiles
// (K-major, or MN-major when a_mn / b_mn is set), issues D = A B^T with
// tcgen05.mma, and dumps all 128 TMEM lanes x N columns of the fp32 accumulator
// so the host can check the layout.
#include <cuda_bf16.h>
#include <stdint.h>

#include "umma.cuh"

using namespace gdn::tc;

// Bytes of one operand tile: K-major rows x ceil(K/64) blocks, or MN-major K rows
// x ceil(rows/64) blocks.
__host__ __device__ inline size_t tile_bytes(int rows, int K, bool mn) {
  return mn ? (size_t)K * 128 * ((rows + 63) / 64) : (size_t)rows * 128 * ((K + 63) / 64);
}

// Stages X [rows x K] (row-major) as a K-major or an MN-major SW128 tile.
__device__ void stage(uint8_t* t, const __nv_bfloat16* X, int rows, int K, bool mn) {
  if (!mn) {
    const int KB = (K + 63) / 64;
    for (int i = threadIdx.x; i < rows * 64 * KB; i += blockDim.x) {
      const int r = i / (64 * KB), k = i % (64 * KB);
      *(__nv_bfloat16*)(t + sw128_offset(r, k, rows)) =
          k < K ? X[r * K + k] : __float2bfloat16(0.f);
    }
  } else {
    for (int i = threadIdx.x; i < rows * K; i += blockDim.x) {
      const int r = i / K, k = i % K;
      *(__nv_bfloat16*)(t + sw128_offset(k, r, K)) = X[r * K + k];
    }
  }
}

__global__ void k_umma_check(const __nv_bfloat16* A, const __nv_bfloat16* B, float* out, int M,
                             int N, int K, int ncols, int a_mn, int b_mn, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = sm;
  uint8_t* sB = sA + tile_bytes(M, K, a_mn);
  uint64_t* bar = (uint64_t*)(sB + tile_bytes(N, K, b_mn));
  uint32_t* tslot = (uint32_t*)(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  stage(sA, A, M, K, a_mn != 0);
  stage(sB, B, N, K, b_mn != 0);
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
    const uint32_t ap = a_mn ? (uint32_t)K * 128u : (uint32_t)M * 128u;
    const uint32_t bp = b_mn ? (uint32_t)K * 128u : (uint32_t)N * 128u;
    mma_tile_x(tmem, smem_u32(sA), a_mn != 0, ap, M, smem_u32(sB), b_mn != 0, bp, N, K, 0u);
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

// Lane layout of the 16x32bx2 TMEM load (tmem_ld16_x2): 4 warps store lane * 1000 +
// column into 128 lanes x 128 columns with 32x32b stores, then read them back with
// tmem_ld16_x2<64> at columns 0, 16, 32, 48.  out[((warp * 32 + t) * 4 + piece) * 16 + j].
__global__ void k_tmem_x2_check(float* out, int* status) {
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // all 512 columns, so that every column the loads can name is allocated
  if (warp == 0) {
    tmem_alloc(&tslot, 512u);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tslot;
  const uint32_t lbase = (uint32_t)(32 * warp) << 16;
  for (int c = 0; c < 128; c += 16) {
    uint32_t r[16];
    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint((float)((32 * warp + lane) * 1000 + c + j));
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(tmem + lbase + c),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  for (int piece = 0; piece < 4; ++piece) {
    float v[16];
    tmem_ld16_x2<64>(tmem + lbase + 16 * piece, v);
    tmem_ld_wait();
    for (int j = 0; j < 16; ++j) out[((warp * 32 + lane) * 4 + piece) * 16 + j] = v[j];
  }
  if (tid == 0) *status = 0;
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512u);
}

extern "C" int tmem_x2_check(float* out, int* status) {
  k_tmem_x2_check<<<1, 128>>>(out, status);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
}

// MN-major operands need M (or N) a multiple of 64 and K a multiple of 16.
extern "C" int umma_check(const void* A, const void* B, float* out, int M, int N, int K,
                          int a_mn, int b_mn, int* status) {
  if ((a_mn && (M % 64 || K % 16)) || (b_mn && (N % 64 || K % 16))) return -3;
  int ncols = 32;
  while (ncols < N) ncols <<= 1;
  // 16 KB of slack after the tiles: every address a descriptor can reach stays
  // inside the allocation whatever the tile layout
  const size_t smem = 1024 + tile_bytes(M, K, a_mn) + tile_bytes(N, K, b_mn) + 64 + 16384;
  cudaFuncSetAttribute(k_umma_check, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_umma_check<<<1, 128, smem>>>((const __nv_bfloat16*)A, (const __nv_bfloat16*)B, out, M, N, K,
                                 ncols, a_mn, b_mn, status);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
}
