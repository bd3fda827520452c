// gdn_decode.cu -- one decode step: every sequence advances its recurrent state by one
// token (the forward at T = 1 per sequence, in its token form).
//
// Gated Delta Networks (Yang et al.) give the per-token update the chunked scan of
// gdn_forward rewrites: with q_hat = q / sqrt(|q|^2 + 1e-6) (k_hat likewise),
// g = exp(-e^{a_log} softplus(alpha + dt_bias)) and beta = sigmoid(beta_raw),
//   delta = beta (v - g S^T k_hat),   S <- g S + k_hat delta^T,   o = scale S^T q_hat.
// A decode step applies it once per (sequence, value head): a state-bound operation
// (the fp32 state is read and written once, Dk Dv FMAs of work per state row pass),
// so it runs on CUDA cores with the state tile staged in shared memory.
#include <cuda_bf16.h>

#include "gdn_device.cuh"
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;   // >= Dv: one thread per value column

struct DecodeParams {
  int Hk, Hv, Dk, Dv, r, head_map;
  float scale;
  const void* q;
  int64_t q_ld;
  const void* k;
  int64_t k_ld;
  const void* v;
  int64_t v_ld;
  const float* alpha;
  int64_t alpha_ld;
  const float* beta_raw;
  int64_t beta_ld;
  const float* a_log;
  const float* dt_bias;
  const float* S_in;
  float* S_out;
  void* o;
  int64_t o_ld;
};

__device__ __forceinline__ float load_io(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_io(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_io(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_io(__nv_bfloat16* p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// One CTA per (sequence n, value head h): the state tile [Dk][Dv] in shared memory
// (16-byte coalesced loads and stores), q_hat and k_hat of the value head's key head
// (h / r, or h % Hk with the modulo head map), then
// thread v forms column v: kv_v = sum_k S[k][v] k_hat[k], delta_v, the new column
// and o_v.  S_in may equal S_out (the tile is read before anything is written).
template <typename T>
__global__ void __launch_bounds__(kDecodeThreads) k_decode(DecodeParams p) {
  extern __shared__ float4 dsm4[];
  float* S = (float*)dsm4;                      // [Dk][Dv]
  float* qs = S + p.Dk * p.Dv;                  // [Dk] q, then q_hat
  float* ks = qs + p.Dk;                        // [Dk] k, then k_hat
  float* red = ks + p.Dk;                       // [2][kDecodeThreads / 32]
  const int n = blockIdx.x, h = blockIdx.y, kh = p.head_map ? h % p.Hk : h / p.r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dk = p.Dk, Dv = p.Dv;
  const size_t SZ = (size_t)Dk * Dv;
  const size_t so = ((size_t)n * p.Hv + h) * SZ;
  const T* q = (const T*)p.q + (int64_t)n * p.q_ld + (int64_t)kh * Dk;
  const T* k = (const T*)p.k + (int64_t)n * p.k_ld + (int64_t)kh * Dk;

  for (int i = tid; i < (int)(SZ / 4); i += kDecodeThreads)
    dsm4[i] = p.S_in ? ((const float4*)(p.S_in + so))[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  float sq = 0.f, sk = 0.f;
  for (int i = tid; i < Dk; i += kDecodeThreads) {
    const float qf = load_io(q, i), kf = load_io(k, i);
    qs[i] = qf;
    ks[i] = kf;
    sq = fmaf(qf, qf, sq);
    sk = fmaf(kf, kf, sk);
  }
  sq = warp_sum(sq);
  sk = warp_sum(sk);
  if (lane == 0) {
    red[warp] = sq;
    red[kDecodeThreads / 32 + warp] = sk;
  }
  __syncthreads();
  float tq = 0.f, tk = 0.f;
#pragma unroll
  for (int w = 0; w < kDecodeThreads / 32; ++w) {
    tq += red[w];
    tk += red[kDecodeThreads / 32 + w];
  }
  const float iq = 1.f / sqrtf(tq + 1e-6f), ik = 1.f / sqrtf(tk + 1e-6f);
  for (int i = tid; i < Dk; i += kDecodeThreads) {
    qs[i] *= iq;
    ks[i] *= ik;
  }
  __syncthreads();
  if (tid < Dv) {
    const int v = tid;
    const float x = p.alpha[(int64_t)n * p.alpha_ld + h] + p.dt_bias[h];
    const float g = expf(-expf(p.a_log[h]) * softplus_f(x));
    const float b = sigmoid_f(p.beta_raw[(int64_t)n * p.beta_ld + h]);
    float kv = 0.f;
    for (int kk = 0; kk < Dk; ++kk) kv = fmaf(S[kk * Dv + v], ks[kk], kv);
    const float d = b * (load_io((const T*)p.v + (int64_t)n * p.v_ld + (int64_t)h * Dv, v) - g * kv);
    float o = 0.f;
    for (int kk = 0; kk < Dk; ++kk) {
      const float s = fmaf(g, S[kk * Dv + v], ks[kk] * d);
      S[kk * Dv + v] = s;
      o = fmaf(s, qs[kk], o);
    }
    store_io((T*)p.o + (int64_t)n * p.o_ld + (int64_t)h * Dv, v, p.scale * o);
  }
  __syncthreads();
  for (int i = tid; i < (int)(SZ / 4); i += kDecodeThreads)
    ((float4*)(p.S_out + so))[i] = dsm4[i];
}

}  // namespace

cudaError_t launch_decode(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                          int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                          int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                          const float* a_log, const float* dt_bias, const float* S_in,
                          float* S_out, void* o, int64_t o_ld, cudaStream_t st) {
  DecodeParams p;
  p.Hk = s->Hk;
  p.Hv = s->Hv;
  p.head_map = s->head_map;
  p.Dk = s->Dk;
  p.Dv = s->Dv;
  p.r = s->Hv / s->Hk;
  p.scale = s->scale > 0.f ? s->scale : 1.f / sqrtf((float)s->Dk);
  p.q = q;
  p.q_ld = q_ld;
  p.k = k;
  p.k_ld = k_ld;
  p.v = v;
  p.v_ld = v_ld;
  p.alpha = alpha;
  p.alpha_ld = alpha_ld;
  p.beta_raw = beta_raw;
  p.beta_ld = beta_ld;
  p.a_log = a_log;
  p.dt_bias = dt_bias;
  p.S_in = S_in;
  p.S_out = S_out;
  p.o = o;
  p.o_ld = o_ld;
  const size_t smem = sizeof(float) * ((size_t)s->Dk * s->Dv + 2 * s->Dk + 2 * kDecodeThreads / 32);
  const dim3 grid((unsigned)s->n_seqs, (unsigned)s->Hv);
  profile_pre(st, KID_DECODE);
  if (s->dtype == GDN_DTYPE_BF16) {
    cudaFuncSetAttribute(k_decode<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    k_decode<__nv_bfloat16><<<grid, kDecodeThreads, smem, st>>>(p);
  } else {
    cudaFuncSetAttribute(k_decode<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_decode<float><<<grid, kDecodeThreads, smem, st>>>(p);
  }
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
