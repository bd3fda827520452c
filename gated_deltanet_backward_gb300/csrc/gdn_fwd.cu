// gdn_fwd.cu -- chunk preparation and the forward state walk.
//
// k_prep       one CTA per (chunk, key head): normalises q and k (L2 with the
//              1e-6 eps inside the square root, lattice-inference gdn_backward.rs
//              gdn_forward_save "L2-normalize q, k"), forms the key Gram K K^T once
//              for the key head, then for each of its v_repeat value heads the gate
//              cumsum G, beta, T = (I + A)^-1, W = T diag(b e^G) K, U = T diag(b) V.
// k_fwd_state  one CTA per (sequence, value head, Dv slice): walks the chunks in
//              order, saving the chunk-start state, forming Delta = U - W S, the
//              output O and the next state.
#include "gdn_device.cuh"

namespace gdn {

template <typename T>
__global__ void __launch_bounds__(kThreads) k_prep(Params p, int write_T) {
  stamp_kept_operands(p);
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, kh = blockIdx.y;
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  const int Dk = p.Dk, Dv = p.Dv, C = kChunk;
  float* Ks = sm;             // [C][Dk] normalised keys
  float* KK = Ks + C * Dk;    // [C][C] K K^T
  float* Tm = KK + C * C;     // [C][C]
  float* A = Tm + C * C;      // [C][C]
  float* gv = A + C * C;      // [C] G
  float* bv = gv + C;         // [C] beta
  float* wv = bv + C;         // [C] beta e^G
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t ck = ((size_t)c * p.Hk + kh) * C;
  for (int row = warp; row < 2 * C; row += kThreads / 32) {
    const bool isk = row >= C;
    const int r = isk ? row - C : row;
    const T* src = (const T*)(isk ? p.k : p.q) + (t0 + r) * (isk ? p.k_ld : p.q_ld) +
                   (int64_t)kh * Dk;
    float* dst = (isk ? p.Kn : p.Qn) + (ck + r) * Dk;
    float ss = 0.f;
    if (r < len)
      for (int i = lane; i < Dk; i += 32) {
        const float x = ldf(src + i);
        ss = fmaf(x, x, ss);
      }
    ss = warp_sum(ss);
    const float nrm = sqrtf(ss + 1e-6f);
    for (int i = lane; i < Dk; i += 32) {
      const float x = r < len ? ldf(src + i) / nrm : 0.f;
      dst[i] = x;
      if (isk) Ks[r * Dk + i] = x;
    }
    if (lane == 0) (isk ? p.nk : p.nq)[ck + r] = nrm;
  }
  __syncthreads();
  block_mm(C, C, Dk, [&](int i, int kk) { return Ks[i * Dk + kk]; },
           [&](int kk, int j) { return Ks[j * Dk + kk]; },
           [&](int i, int j, float acc) { KK[i * C + j] = acc; });
  __syncthreads();
  for (int hh = 0; hh < p.r; ++hh) {
    const int h = value_head(p, kh, hh);
    const size_t ch = (size_t)c * p.Hv + h;
    if (threadIdx.x < C) {
      const int t = threadIdx.x;
      float l = 0.f, b = 0.f;
      if (t < len) {
        b = sigmoid_f(p.beta_raw[(t0 + t) * p.beta_ld + h]);
        const float x = p.alpha[(t0 + t) * p.alpha_ld + h] + p.dt_bias[h];
        l = -expf(p.a_log[h]) * softplus_f(x);
      }
      gv[t] = l;
      bv[t] = b;
    }
    __syncthreads();
    warp0_cumsum64(gv);
    __syncthreads();
    if (threadIdx.x < C) {
      const int t = threadIdx.x;
      wv[t] = bv[t] * expf(gv[t]);
      p.G[ch * C + t] = gv[t];
      p.b[ch * C + t] = bv[t];
    }
    for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
      const int r = idx / C, s = idx % C;
      A[idx] = s < r ? bv[r] * expf(gv[r] - gv[s]) * KK[idx] : 0.f;
    }
    __syncthreads();
    // T = (I + A)^-1 by forward substitution, one row per step.
    for (int r = 0; r < C; ++r) {
      if (threadIdx.x < C) {
        const int j = threadIdx.x;
        float val = 0.f;
        if (j == r) {
          val = 1.f;
        } else if (j < r) {
          float acc = 0.f;
          for (int s = j; s < r; ++s) acc = fmaf(A[r * C + s], Tm[s * C + j], acc);
          val = -acc;
        }
        Tm[r * C + j] = val;
      }
      __syncthreads();
    }
    if (write_T)
      for (int idx = threadIdx.x; idx < C * C; idx += kThreads) p.Tm[ch * C * C + idx] = Tm[idx];
    float* Wd = p.W + ch * C * Dk;
    block_mm(C, Dk, len, [&](int i, int s) { return Tm[i * C + s] * wv[s]; },
             [&](int s, int j) { return Ks[s * Dk + j]; },
             [&](int i, int j, float acc) { Wd[i * Dk + j] = acc; });
    const T* Vs = (const T*)p.v + t0 * p.v_ld + (int64_t)h * Dv;
    float* Ud = p.U + ch * C * Dv;
    block_mm(C, Dv, len, [&](int i, int s) { return Tm[i * C + s] * bv[s]; },
             [&](int s, int j) { return ldf(Vs + (int64_t)s * p.v_ld + j); },
             [&](int i, int j, float acc) { Ud[i * Dv + j] = acc; });
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_fwd_state(Params p, int DVS) {
  extern __shared__ __align__(16) float sm[];
  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * DVS;
  const int kh = key_head(p, h), Dk = p.Dk, Dv = p.Dv, C = kChunk;
  int64_t s0, s1;
  int c0, c1;
  if (!seq_info(p, n, &s0, &s1, &c0, &c1)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, n);
    return;
  }
  float* S = sm;               // [Dk][DVS]
  float* Dl = S + Dk * DVS;    // [C][DVS] Delta
  float* P = Dl + C * DVS;     // [C][C]
  float* gv = P + C * C;       // [C]
  float* ev = gv + C;          // [C] e^G
  float* cv = ev + C;          // [C] e^{G_last - G}
  const size_t SZ = (size_t)Dk * Dv;
  for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
    const int kk = idx / DVS, j = idx % DVS;
    S[idx] = p.S0 ? p.S0[((size_t)n * p.Hv + h) * SZ + (size_t)kk * Dv + v0 + j] : 0.f;
  }
  __syncthreads();
  for (int c = c0; c < c1; ++c) {
    const int64_t t0 = s0 + (int64_t)(c - c0) * C;
    const int len = (int)((s1 - t0) < C ? (s1 - t0) : C);
    const size_t ch = (size_t)c * p.Hv + h;
    if (p.saved) {
      float* sv = p.saved + ch * SZ;
      for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
        const int kk = idx / DVS, j = idx % DVS;
        sv[(size_t)kk * Dv + v0 + j] = S[idx];
      }
    }
    if (threadIdx.x < C) gv[threadIdx.x] = p.G[ch * C + threadIdx.x];
    __syncthreads();
    if (threadIdx.x < C) {
      const int t = threadIdx.x;
      ev[t] = expf(gv[t]);
      cv[t] = t < len ? expf(gv[len - 1] - gv[t]) : 0.f;
    }
    const float* Wc = p.W + ch * C * Dk;
    const float* Uc = p.U + ch * C * Dv + v0;
    const float* Qc = p.Qn + ((size_t)c * p.Hk + kh) * C * Dk;
    const float* Kc = p.Kn + ((size_t)c * p.Hk + kh) * C * Dk;
    // Delta = U - W S
    block_mm(C, DVS, Dk, [&](int i, int kk) { return Wc[i * Dk + kk]; },
             [&](int kk, int j) { return S[kk * DVS + j]; },
             [&](int i, int j, float acc) { Dl[i * DVS + j] = Uc[(size_t)i * Dv + j] - acc; });
    // P = E * (Q K^T), lower triangle including the diagonal
    block_mm(C, C, Dk, [&](int i, int kk) { return Qc[i * Dk + kk]; },
             [&](int kk, int j) { return Kc[j * Dk + kk]; },
             [&](int i, int j, float acc) {
               P[i * C + j] = (j <= i) ? expf(gv[i] - gv[j]) * acc : 0.f;
             });
    __syncthreads();
    // O = scale (diag(e^G) Q S + P Delta)
    T* oc = (T*)p.o + t0 * p.o_ld + (int64_t)h * Dv + v0;
    for (int idx = threadIdx.x; idx < len * DVS; idx += kThreads) {
      const int i = idx / DVS, j = idx % DVS;
      float a1 = 0.f, a2 = 0.f;
      for (int kk = 0; kk < Dk; ++kk) a1 = fmaf(Qc[i * Dk + kk], S[kk * DVS + j], a1);
      for (int s = 0; s <= i; ++s) a2 = fmaf(P[i * C + s], Dl[s * DVS + j], a2);
      stf(oc + (int64_t)i * p.o_ld + j, p.scale * (ev[i] * a1 + a2));
    }
    __syncthreads();
    // S <- e^{G_last} S + K^T diag(c) Delta
    const float eC = expf(gv[len - 1]);
    for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
      const int kk = idx / DVS, j = idx % DVS;
      float acc = 0.f;
      for (int s = 0; s < len; ++s) acc = fmaf(Kc[s * Dk + kk] * cv[s], Dl[s * DVS + j], acc);
      S[idx] = eC * S[idx] + acc;
    }
    __syncthreads();
  }
  if (p.S_T)
    for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
      const int kk = idx / DVS, j = idx % DVS;
      p.S_T[((size_t)n * p.Hv + h) * SZ + (size_t)kk * Dv + v0 + j] = S[idx];
    }
}

static size_t prep_smem(const Params& p) {
  return sizeof(float) * ((size_t)kChunk * p.Dk + 3 * kChunk * kChunk + 3 * kChunk);
}

// fp32 inputs only: bf16 inputs take the tensor-core preparation (launch_prep_tc)
cudaError_t launch_prep(const Params& p, bool write_T, cudaStream_t st) {
  if (p.NC == 0) return cudaSuccess;
  const size_t smem = prep_smem(p);
  dim3 grid(p.NC, p.Hk);
  profile_pre(st, KID_PREP);
  cudaFuncSetAttribute(k_prep<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_prep<float><<<grid, kThreads, smem, st>>>(p, write_T ? 1 : 0);
  profile_post(st);
  return cudaGetLastError();
}

cudaError_t launch_forward(const Params& p, const TmaMaps* maps, cudaStream_t st) {
  const bool bf16 = maps != nullptr;
  if (bf16) {
    // bf16 inputs: tensor-core chunk preparation and state walk
    bool fused = false;
    cudaError_t e = launch_fwd_fused_tc(p, *maps, st, &fused);
    if (e != cudaSuccess) return e;
    if (!fused) {
      e = launch_prep_tc(p, *maps, p.keep != 0, st);
      if (e == cudaSuccess) e = launch_fwd_state_tc(p, st);
      if (e != cudaSuccess) return e;
    }
    // the output from the walks' state and Delta tiles: every unit, or those the fused
    // launch left
    return launch_fwd_out_tc(p, st);
  }
  cudaError_t e = launch_prep(p, p.keep != 0, st);
  if (e != cudaSuccess || p.n_seqs == 0) return e;
  const int DVS = p.Dv < 32 ? p.Dv : 32;
  const size_t smem = sizeof(float) * ((size_t)p.Dk * DVS + (size_t)kChunk * DVS +
                                       kChunk * kChunk + 3 * kChunk);
  dim3 grid(p.n_seqs, p.Hv, p.Dv / DVS);
  profile_pre(st, KID_FWD_STATE);
  cudaFuncSetAttribute(k_fwd_state<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_fwd_state<float><<<grid, kThreads, smem, st>>>(p, DVS);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
