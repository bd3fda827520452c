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
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;

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

// One CTA per (sequence n, value head h, slice of VS value columns): the state columns
// of the slice ([Dk][VS], 16-byte asynchronous copies, all in flight at once) in shared
// memory, q_hat and k_hat of the value head's key head (h / r, or h % Hk with the
// modulo head map), then thread (part, v) of the slice's VS columns and 128 / VS
// row parts forms its share of kv_v = sum_k S[k][v] k_hat[k]; the parts are summed in
// a fixed order, every part updates its rows of column v and adds its share of
// o_v = sum_k S'[k][v] q_hat[k].  Columns are independent, so the slices are too.
// S_in may equal S_out (a CTA reads its slice before it writes it, and no other CTA
// touches it).
template <typename T, int VS>
__global__ void __launch_bounds__(kDecodeThreads) k_decode(DecodeParams p) {
  constexpr int KP = kDecodeThreads / VS;       // row parts
  extern __shared__ float4 dsm4[];
  float* S = (float*)dsm4;                      // [Dk][VS]
  float* qs = S + p.Dk * VS;                    // [Dk] q, then q_hat
  float* ks = qs + p.Dk;                        // [Dk] k, then k_hat
  float* red = ks + p.Dk;                       // [2][kDecodeThreads / 32] norms
  float* part = red + 2 * (kDecodeThreads / 32);  // [KP][VS] partial sums
  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * VS;
  const int kh = p.head_map ? h % p.Hk : h / p.r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dk = p.Dk, Dv = p.Dv;
  const size_t so = ((size_t)n * p.Hv + h) * (size_t)Dk * Dv + v0;   // column v0 of row 0
  const T* q = (const T*)p.q + (int64_t)n * p.q_ld + (int64_t)kh * Dk;
  const T* k = (const T*)p.k + (int64_t)n * p.k_ld + (int64_t)kh * Dk;

  constexpr int C4 = VS / 4;                    // 16-byte pieces of a slice row
  if (p.S_in) {
    for (int i = tid; i < Dk * C4; i += kDecodeThreads)
      tc::cp_async16(dsm4 + i, (const float4*)(p.S_in + so + (size_t)(i / C4) * Dv) + i % C4);
  } else {
    for (int i = tid; i < Dk * C4; i += kDecodeThreads) dsm4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
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
  tc::cp_async_wait_all();   // this thread's share of the slice has landed
  __syncthreads();
  const int vl = tid % VS, kp = tid / VS, v = v0 + vl;
  const int rows = Dk / KP, r0 = kp * rows;
  float kv = 0.f;
  for (int kk = r0; kk < r0 + rows; ++kk) kv = fmaf(S[kk * VS + vl], ks[kk], kv);
  part[kp * VS + vl] = kv;
  __syncthreads();
  kv = 0.f;
#pragma unroll
  for (int j = 0; j < KP; ++j) kv += part[j * VS + vl];
  const float x = p.alpha[(int64_t)n * p.alpha_ld + h] + p.dt_bias[h];
  const float g = expf(-expf(p.a_log[h]) * softplus_f(x));
  const float b = sigmoid_f(p.beta_raw[(int64_t)n * p.beta_ld + h]);
  const float d = b * (load_io((const T*)p.v + (int64_t)n * p.v_ld + (int64_t)h * Dv, v) - g * kv);
  float o = 0.f;
  for (int kk = r0; kk < r0 + rows; ++kk) {
    const float sv = fmaf(g, S[kk * VS + vl], ks[kk] * d);
    S[kk * VS + vl] = sv;
    o = fmaf(sv, qs[kk], o);
  }
  __syncthreads();   // every part has read the kv partials
  part[kp * VS + vl] = o;
  __syncthreads();
  if (kp == 0) {
    o = 0.f;
#pragma unroll
    for (int j = 0; j < KP; ++j) o += part[j * VS + vl];
    store_io((T*)p.o + (int64_t)n * p.o_ld + (int64_t)h * Dv, v, p.scale * o);
  }
  for (int i = tid; i < Dk * C4; i += kDecodeThreads)
    ((float4*)(p.S_out + so + (size_t)(i / C4) * Dv))[i % C4] = dsm4[i];
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
  // slices of 32 value columns (16 for Dv = 16), 128 / VS row parts each
  const int VS = s->Dv >= 32 ? 32 : 16;
  const size_t smem = sizeof(float) * ((size_t)s->Dk * VS + 2 * s->Dk + 2 * kDecodeThreads / 32 +
                                       kDecodeThreads);
  const dim3 grid((unsigned)s->n_seqs, (unsigned)s->Hv, (unsigned)(s->Dv / VS));
  profile_pre(st, KID_DECODE);
  if (s->dtype == GDN_DTYPE_BF16) {
    if (VS == 32)
      k_decode<__nv_bfloat16, 32><<<grid, kDecodeThreads, smem, st>>>(p);
    else
      k_decode<__nv_bfloat16, 16><<<grid, kDecodeThreads, smem, st>>>(p);
  } else {
    if (VS == 32)
      k_decode<float, 32><<<grid, kDecodeThreads, smem, st>>>(p);
    else
      k_decode<float, 16><<<grid, kDecodeThreads, smem, st>>>(p);
  }
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
