// gdn_kda.cu -- the KDA variant in token form, forward and backward: the recurrence with a
// decay gate per key channel instead of one per head.  Channel c of value head h decays by
// g[c] = exp(-exp(a_log[h]) softplus(alpha[t, h*Dk + c] + b_alpha[h*Dk + c])) (the module
// parameters a_log and b_alpha named on the dormouse "KDA attention arm" page), and the
// forward recap's update (lattice-inference 0.6.0, src/attention/gdn_backward.rs) becomes
//   S_d = diag(g) S,  kv = S_d^T k_hat,  delta = beta (v - kv),  S <- S_d + k_hat delta^T,
//   o = scale S^T q_hat.
// The state's value columns evolve independently, so one CTA owns (sequence, value head,
// slice of VS columns) and walks the sequence's tokens in order with its [Dk][VS] slice in
// shared memory.  A sequence of one token is a decode step; longer ones are a prefill in
// token form (one token after another: latency-bound, not the chunked form).  The
// backward (below) walks the same slices in reverse from states saved every few tokens.
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


// ---- backward ----------------------------------------------------------------------------
// Reverse mode of the token form, per (sequence, value head, slice of 32 value columns):
// the columns of S and dS evolve independently, so a slice walks its own dS backwards.
// A forward pass first saves the slice's state before every kKdaCK-th token; then each
// kKdaCK-token segment, last first, is recomputed from its saved state into shared
// memory and walked in reverse:
//   dS += scale q_hat do^T;  dq_hat = scale S_t do;  d delta = dS^T k_hat;  dv = beta d delta
//   d beta = (v - kv) . d delta;  dkv = -beta d delta
//   dk_hat = dS delta + S_d dkv;  dS_d = dS + k_hat dkv^T
//   dg[c] = sum_j S_{t-1}[c][j] dS_d[c][j];  dS = diag(g) dS_d
// dq_hat, dk_hat and dg of a row are sums over all value columns: each slice writes its
// share (a warp's 32 lanes are the slice's 32 columns, so a row's share is a butterfly
// over the warp) and k_kda_bwd_finish adds the slices, then the value heads of a key
// head, in a fixed order.
constexpr int kKdaCK = 8;  // tokens between saved states

struct KdaBwdParams {
  KdaParams f;  // forward arguments (o unused)
  const void* dO;
  int64_t dO_ld;
  const float* dS_T;
  float* dS0;
  void* dv;
  int64_t dv_ld;
  float* ckpt;  // [slots, Hv, Dk, Dv] saved states
  float* part;  // [T, Hv, n_slices, 3 Dk + 1]: dq_hat, dk_hat, dg, d beta shares
  int n_slices;
};

// Saved-state slot of sequence n's k-th segment: floor(begin / CK) + n + k, which no
// other sequence's segment takes.
__device__ __forceinline__ int kda_slot(int t_begin, int n, int k) {
  return t_begin / kKdaCK + n + k;
}

// Sum over the warp's 32 lanes of v[i] for every i < R, left in lane l for i = l % R
// (butterfly reduce-scatter over the low log2(R) lane bits, then an all-reduce over the
// rest).
template <int R>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[R]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = R / 2; s >= 1; s >>= 1) {
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const bool up = (lane & s) != 0;
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  float x = v[0];
#pragma unroll
  for (int m = R; m < 32; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

template <typename T, int R>
__global__ void __launch_bounds__(kKdaThreads) k_kda_bwd(KdaBwdParams b) {
  constexpr int VS = 32, KP = kKdaThreads / VS;  // KP row parts = warps; lanes = columns
  const KdaParams& p = b.f;
  extern __shared__ float4 kda_dyn[];
  float* St = (float*)kda_dyn;                   // [kKdaCK][Dk][VS] states before tokens
  __shared__ float qs[kKdaCK][128], ks[kKdaCK][128], gs[kKdaCK][128];
  __shared__ float kvs[kKdaCK][VS], dls[kKdaCK][VS], vsl[kKdaCK][VS], bets[kKdaCK];
  __shared__ float red[2][kKdaThreads / 32], part_s[KP][VS], ba[128];
  const int n = blockIdx.x, h = blockIdx.y, slice = blockIdx.z, v0 = slice * VS;
  const int kh = p.head_map ? h % p.Hk : h / p.r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Dk = p.Dk, Dv = p.Dv, r0 = warp * R;  // R = Dk / KP rows a thread
  const int t_begin = min(max(__ldg(p.cu + n), 0), p.T);
  const int t_end = min(max(__ldg(p.cu + n + 1), t_begin), p.T);
  const int nseg = (t_end - t_begin + kKdaCK - 1) / kKdaCK;
  const size_t DD = (size_t)Dk * Dv;
  const size_t so = ((size_t)n * p.Hv + h) * DD + v0;
  const float ea = expf(__ldg(p.a_log + h));
  for (int i = tid; i < Dk; i += kKdaThreads) ba[i] = __ldg(p.b_alpha + (int64_t)h * Dk + i);
  const T* vbase = (const T*)p.v + (int64_t)h * Dv + v0 + lane;

  // loads token t's rows into slot j: normalised q, k, the gates, beta and the v column;
  // returns nothing until the block has the norms (two barriers inside)
  auto load_token = [&](int t, int j) {
    float sq = 0.f, sk = 0.f;
    for (int i = tid; i < Dk; i += kKdaThreads) {
      const float qf = to_f(((const T*)p.q)[(int64_t)t * p.q_ld + (int64_t)kh * Dk + i]);
      const float kf = to_f(((const T*)p.k)[(int64_t)t * p.k_ld + (int64_t)kh * Dk + i]);
      qs[j][i] = qf;
      ks[j][i] = kf;
      gs[j][i] = expf(-ea * softplus_f(p.alpha[(int64_t)t * p.alpha_ld + (int64_t)h * Dk + i] + ba[i]));
      sq = fmaf(qf, qf, sq);
      sk = fmaf(kf, kf, sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      red[0][warp] = sq;
      red[1][warp] = sk;
    }
    if (tid < VS) vsl[j][tid] = to_f(vbase[(int64_t)t * p.v_ld - lane + tid]);
    if (tid == 0) bets[j] = sigmoid_f(p.beta_raw[(int64_t)t * p.beta_ld + h]);
    __syncthreads();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int w = 0; w < kKdaThreads / 32; ++w) {
      tq += red[0][w];
      tk += red[1][w];
    }
    const float iq = 1.f / sqrtf(tq + 1e-6f), ik = 1.f / sqrtf(tk + 1e-6f);
    for (int i = tid; i < Dk; i += kKdaThreads) {
      qs[j][i] *= iq;
      ks[j][i] *= ik;
    }
    __syncthreads();
  };
  // one forward token step of the slice held in S (thread: rows r0.., column lane);
  // returns kv and delta of the column; S is updated in place
  auto step = [&](float* S, int j, float& kv, float& dl) {
    float acc = 0.f;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int i = r0 + rr;
      acc = fmaf(gs[j][i] * S[i * VS + lane], ks[j][i], acc);
    }
    part_s[warp][lane] = acc;
    __syncthreads();
    kv = 0.f;
#pragma unroll
    for (int w = 0; w < KP; ++w) kv += part_s[w][lane];
    dl = bets[j] * (vsl[j][lane] - kv);
    __syncthreads();  // part_s is reused
  };

  // ---- forward pass: the state before every kKdaCK-th token goes to its slot
  {
    float S[R];
    for (int rr = 0; rr < R; ++rr)
      S[rr] = p.S_in ? p.S_in[so + (size_t)(r0 + rr) * Dv + lane] : 0.f;
    for (int t = t_begin; t < t_end; ++t) {
      const int k = (t - t_begin) / kKdaCK;
      if ((t - t_begin) % kKdaCK == 0) {
        float* dst = b.ckpt + ((size_t)kda_slot(t_begin, n, k) * p.Hv + h) * DD + v0;
        for (int rr = 0; rr < R; ++rr) dst[(size_t)(r0 + rr) * Dv + lane] = S[rr];
      }
      load_token(t, 0);
      float acc = 0.f;
#pragma unroll
      for (int rr = 0; rr < R; ++rr) acc = fmaf(gs[0][r0 + rr] * S[rr], ks[0][r0 + rr], acc);
      part_s[warp][lane] = acc;
      __syncthreads();
      float kv = 0.f;
#pragma unroll
      for (int w = 0; w < KP; ++w) kv += part_s[w][lane];
      const float dl = bets[0] * (vsl[0][lane] - kv);
#pragma unroll
      for (int rr = 0; rr < R; ++rr) S[rr] = fmaf(gs[0][r0 + rr], S[rr], ks[0][r0 + rr] * dl);
      __syncthreads();  // slot 0 and part_s are reused
    }
  }
  // ---- reverse walk
  float dS[R];
#pragma unroll
  for (int rr = 0; rr < R; ++rr) dS[rr] = b.dS_T ? b.dS_T[so + (size_t)(r0 + rr) * Dv + lane] : 0.f;
  const T* dObase = (const T*)b.dO + (int64_t)h * Dv + v0 + lane;
  T* dvbase = (T*)b.dv + (int64_t)h * Dv + v0 + lane;
  for (int sg = nseg - 1; sg >= 0; --sg) {
    const int ts = t_begin + sg * kKdaCK, len = min(kKdaCK, t_end - ts);
    const float* src = b.ckpt + ((size_t)kda_slot(t_begin, n, sg) * p.Hv + h) * DD + v0;
    for (int rr = 0; rr < R; ++rr)
      St[(r0 + rr) * VS + lane] = src[(size_t)(r0 + rr) * Dv + lane];
    // recompute the segment: St[j] = state before token ts + j
    for (int j = 0; j < len; ++j) {
      load_token(ts + j, j);
      float kv, dl;
      step(St + (size_t)j * Dk * VS, j, kv, dl);
      if (warp == 0) {
        kvs[j][lane] = kv;
        dls[j][lane] = dl;
      }
      if (j + 1 < len) {
        const float* S0j = St + (size_t)j * Dk * VS;
        float* S1j = St + (size_t)(j + 1) * Dk * VS;
        for (int rr = 0; rr < R; ++rr) {
          const int i = r0 + rr;
          S1j[i * VS + lane] = fmaf(gs[j][i], S0j[i * VS + lane], ks[j][i] * dl);
        }
      }
    }
    __syncthreads();
    for (int j = len - 1; j >= 0; --j) {
      const int t = ts + j;
      const float* Sp = St + (size_t)j * Dk * VS;
      const float dov = to_f(dObase[(int64_t)t * b.dO_ld]);
      const float dlt = dls[j][lane], kvv = kvs[j][lane], bet = bets[j];
      float dq_[R], dk_[R], dg_[R];
      float acc = 0.f;
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const int i = r0 + rr;
        const float Stv = fmaf(gs[j][i], Sp[i * VS + lane], ks[j][i] * dlt);
        dS[rr] = fmaf(p.scale * qs[j][i], dov, dS[rr]);
        dq_[rr] = p.scale * Stv * dov;
        acc = fmaf(dS[rr], ks[j][i], acc);
      }
      part_s[warp][lane] = acc;
      __syncthreads();
      float dd = 0.f;
#pragma unroll
      for (int w = 0; w < KP; ++w) dd += part_s[w][lane];
      if (warp == 0) put(dvbase + (int64_t)t * b.dv_ld, bet * dd);
      const float dkv = -bet * dd;
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const int i = r0 + rr;
        const float Spv = Sp[i * VS + lane], Sdv = gs[j][i] * Spv;
        dk_[rr] = fmaf(dS[rr], dlt, Sdv * dkv);
        const float dSd = fmaf(ks[j][i], dkv, dS[rr]);
        dg_[rr] = Spv * dSd;
        dS[rr] = gs[j][i] * dSd;
      }
      float* pt = b.part + (((size_t)t * p.Hv + h) * b.n_slices + slice) * (3 * Dk + 1);
      const float sq_ = warp_reduce_scatter<R>(dq_);
      const float sk_ = warp_reduce_scatter<R>(dk_);
      const float sg_ = warp_reduce_scatter<R>(dg_);
      if (lane < R) {
        pt[r0 + lane] = sq_;
        pt[Dk + r0 + lane] = sk_;
        pt[2 * Dk + r0 + lane] = sg_;
      }
      if (warp == 0) {
        const float db = warp_sum((vsl[j][lane] - kvv) * dd);
        if (lane == 0) pt[3 * Dk] = db;
      }
      __syncthreads();  // part_s is reused
    }
  }
  if (b.dS0)
    for (int rr = 0; rr < R; ++rr) b.dS0[so + (size_t)(r0 + rr) * Dv + lane] = dS[rr];
}

// Per (token t, key head kh): the slices' and value heads' shares added in a fixed order,
// then the L2-norm backward (dq = (dq_hat - q_hat (q_hat . dq_hat)) / |q|) and, per value
// head, the gate backward (dl = dg g, d alpha = dl (-e^{a_log}) sigmoid(x), d beta_raw =
// d beta beta (1 - beta)); dl l goes to lterm for d a_log.
template <typename T>
__global__ void __launch_bounds__(128) k_kda_bwd_finish(KdaBwdParams b, void* dq, int64_t dq_ld,
                                                        void* dk, int64_t dk_ld, float* dalpha,
                                                        int64_t dalpha_ld, float* dbeta,
                                                        int64_t dbeta_ld, float* lterm) {
  const KdaParams& p = b.f;
  const int t = blockIdx.x, kh = blockIdx.y, i = threadIdx.x, Dk = p.Dk;
  __shared__ float red[2][4];
  const bool ok = i < Dk;
  float dqh = 0.f, dkh = 0.f;
  for (int hh = 0; hh < p.r; ++hh) {
    const int h = p.head_map ? kh + hh * p.Hk : kh * p.r + hh;
    const float* pt = b.part + ((size_t)t * p.Hv + h) * b.n_slices * (3 * Dk + 1);
    float dg = 0.f, dbt = 0.f;
    for (int s = 0; s < b.n_slices; ++s) {
      const float* ps = pt + (size_t)s * (3 * Dk + 1);
      if (ok) {
        dqh += ps[i];
        dkh += ps[Dk + i];
        dg += ps[2 * Dk + i];
      }
      dbt += ps[3 * Dk];
    }
    if (ok) {
      const float x = p.alpha[(int64_t)t * p.alpha_ld + (int64_t)h * Dk + i] + p.b_alpha[(int64_t)h * Dk + i];
      const float ea = expf(p.a_log[h]);
      const float l = -ea * softplus_f(x), g = expf(l);
      const float dl = dg * g;
      dalpha[(int64_t)t * dalpha_ld + (int64_t)h * Dk + i] = dl * (-ea) * sigmoid_f(x);
      lterm[((size_t)t * p.Hv + h) * Dk + i] = dl * l;
    }
    if (i == 0) {
      const float be = sigmoid_f(p.beta_raw[(int64_t)t * p.beta_ld + h]);
      dbeta[(int64_t)t * dbeta_ld + h] = dbt * be * (1.f - be);
    }
  }
  const T* qr = (const T*)p.q + (int64_t)t * p.q_ld + (int64_t)kh * Dk;
  const T* kr = (const T*)p.k + (int64_t)t * p.k_ld + (int64_t)kh * Dk;
  const float qf = ok ? to_f(qr[i]) : 0.f, kf = ok ? to_f(kr[i]) : 0.f;
  float a0 = warp_sum(qf * qf), a1 = warp_sum(kf * kf);
  if ((i & 31) == 0) {
    red[0][i >> 5] = a0;
    red[1][i >> 5] = a1;
  }
  __syncthreads();
  const float nq = sqrtf(red[0][0] + red[0][1] + red[0][2] + red[0][3] + 1e-6f);
  const float nk = sqrtf(red[1][0] + red[1][1] + red[1][2] + red[1][3] + 1e-6f);
  const float qh = qf / nq, kh_ = kf / nk;
  __syncthreads();
  a0 = warp_sum(qh * dqh);
  a1 = warp_sum(kh_ * dkh);
  if ((i & 31) == 0) {
    red[0][i >> 5] = a0;
    red[1][i >> 5] = a1;
  }
  __syncthreads();
  const float dotq = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  const float dotk = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  if (ok) {
    put((T*)dq + (int64_t)t * dq_ld + (int64_t)kh * Dk + i, (dqh - qh * dotq) / nq);
    put((T*)dk + (int64_t)t * dk_ld + (int64_t)kh * Dk + i, (dkh - kh_ * dotk) / nk);
  }
}

// d b_alpha[j] = sum_t dalpha[t, j] and colsum[j] = sum_t lterm[t, j], t in order, one
// thread per column j of Hv Dk; then d a_log[h] = sum of colsum over the head's columns.
__global__ void __launch_bounds__(256) k_kda_bwd_sums(const float* dalpha, int64_t dalpha_ld,
                                                      const float* lterm, int T, int n,
                                                      float* db_alpha, float* colsum) {
  const int j = blockIdx.x * 256 + threadIdx.x;
  if (j >= n) return;
  float a = 0.f, c = 0.f;
  for (int t = 0; t < T; ++t) {
    a += dalpha[(int64_t)t * dalpha_ld + j];
    c += lterm[(size_t)t * n + j];
  }
  db_alpha[j] = a;
  colsum[j] = c;
}
__global__ void __launch_bounds__(128) k_kda_bwd_alog(const float* colsum, int Dk, float* da_log) {
  const int h = blockIdx.x;
  __shared__ float red[4];
  float s = 0.f;
  for (int i = threadIdx.x; i < Dk; i += 128) s += colsum[(size_t)h * Dk + i];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) da_log[h] = red[0] + red[1] + red[2] + red[3];
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

namespace gdn {

size_t kda_bwd_workspace_floats(const gdn_shape* s) {
  const size_t T = (size_t)s->total_tokens, Hv = s->Hv, Dk = s->Dk, Dv = s->Dv;
  const size_t slots = T / kKdaCK + (size_t)s->n_seqs + 1;
  const size_t n_slices = Dv / 32;
  return slots * Hv * Dk * Dv                  // saved states
         + T * Hv * n_slices * (3 * Dk + 1)    // per-slice shares
         + T * Hv * Dk                         // dl * l per token
         + Hv * Dk + 64;                       // column sums
}

cudaError_t launch_kda_backward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                                int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                                int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                                const float* a_log, const float* b_alpha, const int32_t* cu,
                                const float* S0, const void* dO, int64_t dO_ld,
                                const float* dS_T, void* dq, int64_t dq_ld, void* dk,
                                int64_t dk_ld, void* dv, int64_t dv_ld, float* dalpha,
                                int64_t dalpha_ld, float* dbeta, int64_t dbeta_ld, float* da_log,
                                float* db_alpha, float* dS0, float* ws, cudaStream_t st) {
  KdaBwdParams b;
  KdaParams& p = b.f;
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
  p.S_in = S0;
  p.S_out = nullptr;
  p.o = nullptr;
  p.o_ld = 0;
  b.dO = dO;
  b.dO_ld = dO_ld;
  b.dS_T = dS_T;
  b.dS0 = dS0;
  b.dv = dv;
  b.dv_ld = dv_ld;
  b.n_slices = s->Dv / 32;
  const size_t T = (size_t)s->total_tokens, Hv = s->Hv, Dk = s->Dk, Dv = s->Dv;
  const size_t slots = T / kKdaCK + (size_t)s->n_seqs + 1;
  b.ckpt = ws;
  b.part = b.ckpt + slots * Hv * Dk * Dv;
  float* lterm = b.part + T * Hv * b.n_slices * (3 * Dk + 1);
  float* colsum = lterm + T * Hv * Dk;
  const size_t smem = sizeof(float) * (size_t)kKdaCK * Dk * 32;
  const dim3 grid((unsigned)s->n_seqs, (unsigned)s->Hv, (unsigned)b.n_slices);
  const bool bf = s->dtype == GDN_DTYPE_BF16;
  cudaError_t e = cudaSuccess;
  profile_pre(st, KID_KDA_BWD);
#define GDN_KDA_BWD(TT, RR)                                                                  \
  {                                                                                          \
    static bool attr = false;                                                                \
    if (!attr) {                                                                             \
      e = cudaFuncSetAttribute(k_kda_bwd<TT, RR>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                               (int)smem);                                                   \
      attr = e == cudaSuccess;                                                               \
    }                                                                                        \
    if (e == cudaSuccess) k_kda_bwd<TT, RR><<<grid, kKdaThreads, smem, st>>>(b);             \
  }
  switch (s->Dk / 4) {
    case 4:
      if (bf) GDN_KDA_BWD(__nv_bfloat16, 4) else GDN_KDA_BWD(float, 4)
      break;
    case 8:
      if (bf) GDN_KDA_BWD(__nv_bfloat16, 8) else GDN_KDA_BWD(float, 8)
      break;
    case 16:
      if (bf) GDN_KDA_BWD(__nv_bfloat16, 16) else GDN_KDA_BWD(float, 16)
      break;
    case 32:
      if (bf) GDN_KDA_BWD(__nv_bfloat16, 32) else GDN_KDA_BWD(float, 32)
      break;
    default: e = cudaErrorInvalidValue;
  }
#undef GDN_KDA_BWD
  profile_post(st);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (T > 0) {
    profile_pre(st, KID_KDA_BWD);
    const dim3 g2((unsigned)T, (unsigned)s->Hk);
    if (bf)
      k_kda_bwd_finish<__nv_bfloat16><<<g2, 128, 0, st>>>(b, dq, dq_ld, dk, dk_ld, dalpha, dalpha_ld,
                                                          dbeta, dbeta_ld, lterm);
    else
      k_kda_bwd_finish<float><<<g2, 128, 0, st>>>(b, dq, dq_ld, dk, dk_ld, dalpha, dalpha_ld, dbeta,
                                                  dbeta_ld, lterm);
    profile_post(st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int ncol = (int)(Hv * Dk);
  profile_pre(st, KID_SUM_PARTS);
  k_kda_bwd_sums<<<(ncol + 255) / 256, 256, 0, st>>>(dalpha, dalpha_ld, lterm, (int)T, ncol,
                                                     db_alpha, colsum);
  k_kda_bwd_alog<<<(unsigned)Hv, 128, 0, st>>>(colsum, (int)Dk, da_log);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
