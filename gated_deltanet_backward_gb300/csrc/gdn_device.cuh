// gdn_device.cuh -- device helpers shared by the forward and backward kernels.
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Record the first device-side error; later ones keep the first.
__device__ __forceinline__ void set_status(DeviceStatus* st, int code, int detail) {
  if (atomicCAS(&st->code, 0, code) == 0) st->detail = detail;
}

// A reusing backward whose workspace does not carry this shape's tag records
// GDN_ERR_NOT_KEPT and does nothing.  Every backward kernel asks first.
__device__ __forceinline__ bool kept_operands_missing(const Params& p) {
  if (!p.reuse) return false;
  if (*(volatile const uint32_t*)&p.status->tag == p.tag) return false;
  if (threadIdx.x == 0) set_status(p.status, GDN_ERR_NOT_KEPT, 0);
  return true;
}

// The first CTA of a keeping forward's preparation stamps the workspace.
__device__ __forceinline__ void stamp_kept_operands(const Params& p) {
  if (p.keep && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) p.status->tag = p.tag;
}

// softplus(x) = log(1 + e^x) in the overflow-free form max(x,0) + log1p(e^-|x|).
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// Locates global chunk c: its sequence n, first token t0 and length len.
// Returns false (and the caller records GDN_ERR_DEVICE_BOUNDS) when
// cu_seqlens / chunk_offsets do not describe chunk c consistently.
__device__ __forceinline__ bool chunk_info_at(const int32_t* cu, const int32_t* coff, int n_seqs,
                                              int NC, int64_t T, int c, int* n_out, int64_t* t0,
                                              int* len) {
  if (n_seqs <= 0 || c < 0 || c >= NC) return false;
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (coff[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const int n = lo;
  const int j = c - coff[n];
  const int64_t s = cu[n], e = cu[n + 1];
  const int64_t start = s + (int64_t)j * kChunk;
  if (j < 0 || c >= coff[n + 1] || s < 0 || e < s || e > T || start >= e) return false;
  *n_out = n;
  *t0 = start;
  *len = (int)((e - start) < kChunk ? (e - start) : kChunk);
  return true;
}
// chunk_info_at on the batch's own cu_seqlens / chunk_offsets (global memory)
__device__ __forceinline__ bool chunk_info(const Params& p, int c, int* n_out, int64_t* t0,
                                           int* len) {
  return chunk_info_at(p.cu, p.coff, p.n_seqs, p.NC, p.T, c, n_out, t0, len);
}

// Checks that sequence n's chunk range matches its token range.
__device__ __forceinline__ bool seq_info(const Params& p, int n, int64_t* s, int64_t* e, int* c0,
                                         int* c1) {
  *s = p.cu[n];
  *e = p.cu[n + 1];
  *c0 = p.coff[n];
  *c1 = p.coff[n + 1];
  const int64_t want = (*e - *s + kChunk - 1) / kChunk;
  return *s >= 0 && *e >= *s && *e <= p.T && *c0 >= 0 && *c1 <= p.NC && (*c1 - *c0) == want;
}

// Block-wide small contraction: for i < M, j < N,
//   out(i, j, sum_{kk < K} a(i, kk) * b(kk, j)).
// Consecutive threads take consecutive j.  fp32 FMA on the CUDA cores.
template <class FA, class FB, class FO>
__device__ __forceinline__ void block_mm(int M, int N, int K, FA a, FB b, FO out) {
  for (int idx = threadIdx.x; idx < M * N; idx += blockDim.x) {
    const int i = idx / N, j = idx - (idx / N) * N;
    float acc = 0.f;
    for (int kk = 0; kk < K; ++kk) acc = fmaf(a(i, kk), b(kk, j), acc);
    out(i, j, acc);
  }
}

// Inclusive prefix sum of x[0..63] in place, by warp 0 (two values per lane).
__device__ __forceinline__ void warp0_cumsum64(float* x) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float a = x[2 * lane], b = a + x[2 * lane + 1];
    float run = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += y;
    }
    const float before = run - b;
    x[2 * lane] = before + a;
    x[2 * lane + 1] = run;
  }
}

}  // namespace gdn
