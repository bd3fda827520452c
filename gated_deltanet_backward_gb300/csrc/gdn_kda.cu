// gdn_kda.cu -- the KDA variant's forward in token form: the recurrence with a decay gate
// per key channel instead of one per head.  Channel c of value head h decays by
// g[c] = exp(-exp(a_log[h]) softplus(alpha[t, h*Dk + c] + b_alpha[h*Dk + c])) (the module
// parameters a_log and b_alpha named on the dormouse "KDA attention arm" page), and the
// forward recap's update (lattice-inference 0.6.0, src/attention/gdn_backward.rs) becomes
//   S_d = diag(g) S,  kv = S_d^T k_hat,  delta = beta (v - kv),  S <- S_d + k_hat delta^T,
//   o = scale S^T q_hat.
// The state's value columns evolve independently, so one CTA owns (sequence, value head,
// slice of VS columns) and walks the sequence's tokens in order with its [Dk][VS] slice in
// shared memory.  A sequence of one token is a decode step; longer ones are a prefill in
// token form (one token after another: latency-bound, not the chunked form).
#include <cuda_bf16.h>

#include "gdn_device.cuh"
#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kKdaThreads = 128;

struct KdaParams {
  int Hk, Hv, Dk, Dv, r, head_map, n_seqs, T;
  float scale;
  const void* q;
  int64_t q_ld;
  const void* k;
  int64_t k_ld;
  const void* v;
  int64_t v_ld;
  const float* alpha;  // [T, alpha_ld >= Hv*Dk]
  int64_t alpha_ld;
  const float* beta_raw;
  int64_t beta_ld;
  const float* a_log;    // [Hv]
  const float* b_alpha;  // [Hv*Dk]
  const int32_t* cu;
  const float* S_in;
  float* S_out;
  void* o;
  int64_t o_ld;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void put(float* p, float x) { *p = x; }
__device__ __forceinline__ void put(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Raw rows of one token, staged by cp.async one token ahead.
template <typename T>
struct KdaStage {
  T q[128], k[128];
  float alpha[128];
  T v[32];
  float beta;
  float pad[3];
};

template <typename T, int VS>
__global__ void __launch_bounds__(kKdaThreads) k_kda_fwd(KdaParams p) {
  constexpr int KP = kKdaThreads / VS;  // row parts
  __shared__ KdaStage<T> stg[2];
  __shared__ float qs[128], ks[128], gs[128], ba[128];
  __shared__ float red[2][kKdaThreads / 32];
  __shared__ float part[KP][VS];
  extern __shared__ float4 kda_dyn[];
  float* S = (float*)kda_dyn;  // [Dk][VS]
  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * VS;
  const int kh = p.head_map ? h % p.Hk : h / p.r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dk = p.Dk, Dv = p.Dv;
  // the sequence's tokens, clamped to [0, T): a malformed cu_seqlens never moves a load
  const int t_begin = min(max(__ldg(p.cu + n), 0), p.T);
  const int t_end = min(max(__ldg(p.cu + n + 1), t_begin), p.T);
  const size_t so = ((size_t)n * p.Hv + h) * (size_t)Dk * Dv + v0;
  constexpr int C4 = VS / 4;
  if (p.S_in) {
    for (int i = tid; i < Dk * C4; i += kKdaThreads)
      tc::cp_async16(kda_dyn + i, (const float4*)(p.S_in + so + (size_t)(i / C4) * Dv) + i % C4);
  } else {
    for (int i = tid; i < Dk * C4; i += kKdaThreads) kda_dyn[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float ea = expf(__ldg(p.a_log + h));
  for (int i = tid; i < Dk; i += kKdaThreads) ba[i] = __ldg(p.b_alpha + (int64_t)h * Dk + i);
  // stage token t's rows into stg[b] (4-byte copies; element counts are even)
  auto stage = [&](int t, int b) {
    if (t >= t_end) return;
    constexpr int E = 4 / (int)sizeof(T);  // elements per 4-byte copy
    const T* qr = (const T*)p.q + (int64_t)t * p.q_ld + (int64_t)kh * Dk;
    const T* kr = (const T*)p.k + (int64_t)t * p.k_ld + (int64_t)kh * Dk;
    const T* vr = (const T*)p.v + (int64_t)t * p.v_ld + (int64_t)h * Dv + v0;
    const float* ar = p.alpha + (int64_t)t * p.alpha_ld + (int64_t)h * Dk;
    const int nq = Dk / E, nv = VS / E;
    for (int i = tid; i < 2 * nq + Dk + nv + 1; i += kKdaThreads) {
      if (i < nq)
        tc::cp_async4(stg[b].q + i * E, qr + i * E);
      else if (i < 2 * nq)
        tc::cp_async4(stg[b].k + (i - nq) * E, kr + (i - nq) * E);
      else if (i < 2 * nq + Dk)
        tc::cp_async4(stg[b].alpha + (i - 2 * nq), ar + (i - 2 * nq));
      else if (i < 2 * nq + Dk + nv)
        tc::cp_async4(stg[b].v + (i - 2 * nq - Dk) * E, vr + (i - 2 * nq - Dk) * E);
      else if (i == 2 * nq + Dk + nv)
        tc::cp_async4(&stg[b].beta, p.beta_raw + (int64_t)t * p.beta_ld + h);
    }
  };
  stage(t_begin, 0);
  tc::cp_async_commit();
  const int vl = tid % VS, kp = tid / VS;
  const int rows = Dk / KP, r0 = kp * rows;
  for (int t = t_begin; t < t_end; ++t) {
    const int b = (t - t_begin) & 1;
    stage(t + 1, b ^ 1);  // the buffer read two tokens ago
    tc::cp_async_commit();
    tc::cp_async_wait<1>();  // this token's rows (and, the first time, the state) landed
    __syncthreads();
    float sq = 0.f, sk = 0.f;
    for (int i = tid; i < Dk; i += kKdaThreads) {
      const float qf = to_f(stg[b].q[i]), kf = to_f(stg[b].k[i]);
      qs[i] = qf;
      ks[i] = kf;
      gs[i] = expf(-ea * softplus_f(stg[b].alpha[i] + ba[i]));
      sq = fmaf(qf, qf, sq);
      sk = fmaf(kf, kf, sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      red[0][warp] = sq;
      red[1][warp] = sk;
    }
    __syncthreads();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int w = 0; w < kKdaThreads / 32; ++w) {
      tq += red[0][w];
      tk += red[1][w];
    }
    const float iq = 1.f / sqrtf(tq + 1e-6f), ik = 1.f / sqrtf(tk + 1e-6f);
    // kv_v = sum_k g_k S[k][v] k_hat_k, by row parts then in a fixed order
    float kv = 0.f;
    for (int kk = r0; kk < r0 + rows; ++kk) kv = fmaf(gs[kk] * S[kk * VS + vl], ks[kk], kv);
    part[kp][vl] = kv * ik;
    __syncthreads();
    kv = 0.f;
#pragma unroll
    for (int j = 0; j < KP; ++j) kv += part[j][vl];
    const float beta = sigmoid_f(stg[b].beta);
    const float d = beta * (to_f(stg[b].v[vl]) - kv);
    float o = 0.f;
    for (int kk = r0; kk < r0 + rows; ++kk) {
      const float sv = fmaf(gs[kk], S[kk * VS + vl], ks[kk] * ik * d);
      S[kk * VS + vl] = sv;
      o = fmaf(sv, qs[kk], o);
    }
    __syncthreads();  // every part has read the kv partials
    part[kp][vl] = o * iq;
    __syncthreads();
    if (kp == 0) {
      o = 0.f;
#pragma unroll
      for (int j = 0; j < KP; ++j) o += part[j][vl];
      put((T*)p.o + (int64_t)t * p.o_ld + (int64_t)h * Dv + v0 + vl, p.scale * o);
    }
  }
  tc::cp_async_wait<0>();
  __syncthreads();
  for (int i = tid; i < Dk * C4; i += kKdaThreads)
    ((float4*)(p.S_out + so + (size_t)(i / C4) * Dv))[i % C4] = kda_dyn[i];
}

}  // namespace

cudaError_t launch_kda_forward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                               int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                               int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                               const float* a_log, const float* b_alpha, const int32_t* cu,
                               const float* S_in, float* S_out, void* o, int64_t o_ld,
                               cudaStream_t st) {
  KdaParams p;
  p.Hk = s->Hk;
  p.Hv = s->Hv;
  p.Dk = s->Dk;
  p.Dv = s->Dv;
  p.r = s->Hv / s->Hk;
  p.head_map = s->head_map;
  p.n_seqs = s->n_seqs;
  p.T = (int)s->total_tokens;
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
  p.b_alpha = b_alpha;
  p.cu = cu;
  p.S_in = S_in;
  p.S_out = S_out;
  p.o = o;
  p.o_ld = o_ld;
  const int VS = s->Dv >= 32 ? 32 : 16;
  const size_t smem = sizeof(float) * (size_t)s->Dk * VS;
  const dim3 grid((unsigned)s->n_seqs, (unsigned)s->Hv, (unsigned)(s->Dv / VS));
  profile_pre(st, KID_KDA_FWD);
  if (s->dtype == GDN_DTYPE_BF16) {
    if (VS == 32)
      k_kda_fwd<__nv_bfloat16, 32><<<grid, kKdaThreads, smem, st>>>(p);
    else
      k_kda_fwd<__nv_bfloat16, 16><<<grid, kKdaThreads, smem, st>>>(p);
  } else {
    if (VS == 32)
      k_kda_fwd<float, 32><<<grid, kKdaThreads, smem, st>>>(p);
    else
      k_kda_fwd<float, 16><<<grid, kKdaThreads, smem, st>>>(p);
  }
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
