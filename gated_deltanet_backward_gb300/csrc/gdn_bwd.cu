// gdn_bwd.cu -- the reverse chunk walk and the per-chunk gradients.
//
// Reverse-mode derivative of the chunked form in gdn_internal.cuh; per chunk,
// given dO and dS = dL/dS_next (the adjoint carried from the chunk after):
//   dDelta  = scale P^T dO + diag(c) K dS
//   dS_prev = e^{G_last} dS + scale Q^T diag(e^G) dO - W^T dDelta
// (k_bwd_state, sequential over chunks), then, independently per chunk
// (k_bwd_grads), dQ, dK, dV, d beta, dG through P, E, T = (I+A)^-1, W and U, and
// the gate / sigmoid / L2-norm epilogues of lattice-inference gdn_backward.rs
// section 4 (steps 4e, 4f, 4h).  dq/dk of a key head are summed over its value
// heads in ascending head order (k_bwd_qk), and d a_log / d dt_bias over the
// chunks in ascending chunk order (k_bwd_gates): no atomics on the data path,
// so every output is bit-reproducible.
#include "gdn_device.cuh"

namespace gdn {

template <typename T>
__global__ void __launch_bounds__(kThreads) k_bwd_state(Params p, int DVS) {
  if (kept_operands_missing(p)) return;
  extern __shared__ __align__(16) float sm[];
  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * DVS;
  const int kh = key_head(p, h), Dk = p.Dk, Dv = p.Dv, C = kChunk;
  int64_t s0, s1;
  int c0, c1;
  if (!seq_info(p, n, &s0, &s1, &c0, &c1)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, n);
    return;
  }
  float* dS = sm;              // [Dk][DVS]
  float* dD = dS + Dk * DVS;   // [C][DVS] d Delta
  float* P = dD + C * DVS;     // [C][C]
  float* gv = P + C * C;       // [C]
  float* ev = gv + C;          // [C]
  float* cv = ev + C;          // [C]
  const size_t SZ = (size_t)Dk * Dv;
  for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
    const int kk = idx / DVS, j = idx % DVS;
    dS[idx] = p.dS_T ? p.dS_T[((size_t)n * p.Hv + h) * SZ + (size_t)kk * Dv + v0 + j] : 0.f;
  }
  __syncthreads();
  for (int c = c1 - 1; c >= c0; --c) {
    const int64_t t0 = s0 + (int64_t)(c - c0) * C;
    const int len = (int)((s1 - t0) < C ? (s1 - t0) : C);
    const size_t ch = (size_t)c * p.Hv + h;
    float* dsv = p.dS + ch * SZ;
    for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
      const int kk = idx / DVS, j = idx % DVS;
      dsv[(size_t)kk * Dv + v0 + j] = dS[idx];
    }
    if (threadIdx.x < C) gv[threadIdx.x] = p.G[ch * C + threadIdx.x];
    __syncthreads();
    if (threadIdx.x < C) {
      const int t = threadIdx.x;
      ev[t] = expf(gv[t]);
      cv[t] = t < len ? expf(gv[len - 1] - gv[t]) : 0.f;
    }
    const float* Wc = p.W + ch * C * Dk;
    const float* Qc = p.Qn + ((size_t)c * p.Hk + kh) * C * Dk;
    const float* Kc = p.Kn + ((size_t)c * p.Hk + kh) * C * Dk;
    const T* dOc = (const T*)p.dO + t0 * p.dO_ld + (int64_t)h * Dv + v0;
    block_mm(C, C, Dk, [&](int i, int kk) { return Qc[i * Dk + kk]; },
             [&](int kk, int j) { return Kc[j * Dk + kk]; },
             [&](int i, int j, float acc) {
               P[i * C + j] = (j <= i && i < len) ? expf(gv[i] - gv[j]) * acc : 0.f;
             });
    __syncthreads();
    // dDelta = scale P^T dO + diag(c) K dS
    float* dDg = p.dD + ch * C * Dv + v0;
    for (int idx = threadIdx.x; idx < C * DVS; idx += kThreads) {
      const int s = idx / DVS, j = idx % DVS;
      float val = 0.f;
      if (s < len) {
        float a1 = 0.f, a2 = 0.f;
        for (int r = s; r < len; ++r) a1 = fmaf(P[r * C + s], ldf(dOc + (int64_t)r * p.dO_ld + j), a1);
        for (int kk = 0; kk < Dk; ++kk) a2 = fmaf(Kc[s * Dk + kk], dS[kk * DVS + j], a2);
        val = p.scale * a1 + cv[s] * a2;
      }
      dD[idx] = val;
      dDg[(size_t)s * Dv + j] = val;
    }
    __syncthreads();
    // dS <- e^{G_last} dS + scale Q^T diag(e^G) dO - W^T dDelta
    const float eC = expf(gv[len - 1]);
    for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
      const int kk = idx / DVS, j = idx % DVS;
      float a1 = 0.f, a2 = 0.f;
      for (int r = 0; r < len; ++r) {
        a1 = fmaf(Qc[r * Dk + kk] * ev[r], ldf(dOc + (int64_t)r * p.dO_ld + j), a1);
        a2 = fmaf(Wc[r * Dk + kk], dD[r * DVS + j], a2);
      }
      dS[idx] = eC * dS[idx] + p.scale * a1 - a2;
    }
    __syncthreads();
  }
  if (p.dS0)
    for (int idx = threadIdx.x; idx < Dk * DVS; idx += kThreads) {
      const int kk = idx / DVS, j = idx % DVS;
      p.dS0[((size_t)n * p.Hv + h) * SZ + (size_t)kk * Dv + v0 + j] = dS[idx];
    }
}

// Per (chunk, value head) gradients.  dQ_hat / dK_hat of this value head go to
// the dQh / dKh workspace partials; k_bwd_qk sums them per key head.
template <typename T>
__global__ void __launch_bounds__(kThreads) k_bwd_grads(Params p) {
  if (kept_operands_missing(p)) return;
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, h = blockIdx.y, kh = key_head(p, h);
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  const int Dk = p.Dk, Dv = p.Dv, C = kChunk, Dm = Dk > Dv ? Dk : Dv;
  float* Dl = sm;               // [C][Dv] Delta
  float* dW = Dl + C * Dv;      // [C][Dk]
  float* Tmp = dW + C * Dk;     // [C][Dm]
  float* KK = Tmp + C * Dm;     // [C][C]
  float* E = KK + C * C;        // [C][C] exp(G_r - G_s), s <= r
  float* Pm = E + C * C;        // [C][C]
  float* dP = Pm + C * C;       // [C][C]; later dA
  float* dT = dP + C * C;       // [C][C]
  float* X = dT + C * C;        // [C][C]
  float* gv = X + C * C;        // [C] G
  float* ev = gv + C;           // [C] e^G
  float* cv = ev + C;           // [C] e^{G_last - G}
  float* bv = cv + C;           // [C] beta
  float* dG = bv + C;           // [C]
  float* db = dG + C;           // [C]
  float* red = db + C;          // [kThreads / 32] block reduction scratch
  const size_t ch = (size_t)c * p.Hv + h;
  const size_t SZ = (size_t)Dk * Dv;
  const float* S = p.saved_in + ch * SZ;
  const float* dSg = p.dS + ch * SZ;
  const float* Wc = p.W + ch * C * Dk;
  const float* Uc = p.U + ch * C * Dv;
  const float* Tc = p.Tm + ch * C * C;
  const float* dDc = p.dD + ch * C * Dv;
  const float* Qc = p.Qn + ((size_t)c * p.Hk + kh) * C * Dk;
  const float* Kc = p.Kn + ((size_t)c * p.Hk + kh) * C * Dk;
  const T* dOc = (const T*)p.dO + t0 * p.dO_ld + (int64_t)h * Dv;
  const T* Vc = (const T*)p.v + t0 * p.v_ld + (int64_t)h * Dv;
  float* dQh = p.dQh + ch * C * Dk;
  float* dKh = p.dKh + ch * C * Dk;
  auto dO_at = [&](int r, int j) { return r < len ? ldf(dOc + (int64_t)r * p.dO_ld + j) : 0.f; };
  auto V_at = [&](int s, int j) { return s < len ? ldf(Vc + (int64_t)s * p.v_ld + j) : 0.f; };

  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    gv[t] = p.G[ch * C + t];
    bv[t] = p.b[ch * C + t];
    dG[t] = 0.f;
    db[t] = 0.f;
  }
  __syncthreads();
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    ev[t] = expf(gv[t]);
    cv[t] = t < len ? expf(gv[len - 1] - gv[t]) : 0.f;
  }
  // Delta = U - W S
  block_mm(C, Dv, Dk, [&](int i, int kk) { return Wc[i * Dk + kk]; },
           [&](int kk, int j) { return S[(size_t)kk * Dv + j]; },
           [&](int i, int j, float acc) { Dl[i * Dv + j] = Uc[i * Dv + j] - acc; });
  block_mm(C, C, Dk, [&](int i, int kk) { return Kc[i * Dk + kk]; },
           [&](int kk, int j) { return Kc[j * Dk + kk]; },
           [&](int i, int j, float acc) { KK[i * C + j] = acc; });
  block_mm(C, C, Dk, [&](int i, int kk) { return Qc[i * Dk + kk]; },
           [&](int kk, int j) { return Kc[j * Dk + kk]; },
           [&](int i, int j, float acc) {
             const float e = j <= i ? expf(gv[i] - gv[j]) : 0.f;
             E[i * C + j] = e;
             Pm[i * C + j] = e * acc;
           });
  __syncthreads();
  // dP = scale (dO Delta^T), lower triangle including the diagonal, valid rows
  block_mm(C, C, Dv, [&](int i, int j) { return dO_at(i, j); },
           [&](int j, int s) { return Dl[s * Dv + j]; },
           [&](int i, int s, float acc) { dP[i * C + s] = (s <= i) ? p.scale * acc : 0.f; });
  __syncthreads();
  // dQ_hat = scale diag(e^G) dO S^T + (dP * E) K
  for (int idx = threadIdx.x; idx < C * Dk; idx += kThreads) {
    const int r = idx / Dk, kk = idx % Dk;
    float a1 = 0.f, a2 = 0.f;
    if (r < len) {
      for (int j = 0; j < Dv; ++j) a1 = fmaf(dO_at(r, j), S[(size_t)kk * Dv + j], a1);
      for (int s = 0; s <= r; ++s) a2 = fmaf(dP[r * C + s] * E[r * C + s], Kc[s * Dk + kk], a2);
    }
    dQh[idx] = p.scale * ev[r] * a1 + a2;
  }
  // dK_hat = (dP * E)^T Q + diag(c) Delta dS^T
  for (int idx = threadIdx.x; idx < C * Dk; idx += kThreads) {
    const int s = idx / Dk, kk = idx % Dk;
    float a1 = 0.f, a2 = 0.f;
    for (int r = s; r < len; ++r) a1 = fmaf(dP[r * C + s] * E[r * C + s], Qc[r * Dk + kk], a1);
    for (int j = 0; j < Dv; ++j) a2 = fmaf(Dl[s * Dv + j], dSg[(size_t)kk * Dv + j], a2);
    dKh[idx] = a1 + cv[s] * a2;
  }
  // dG from P: dG_r += sum_s (dP*P)_rs, dG_s -= sum_r (dP*P)_rs
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float rs = 0.f, cs = 0.f;
    for (int s = 0; s < C; ++s) rs += dP[t * C + s] * Pm[t * C + s];
    for (int r = 0; r < C; ++r) cs += dP[r * C + t] * Pm[r * C + t];
    dG[t] += rs - cs;
  }
  // Tmp = (Q S) * dO  ->  dG_r += scale e^{G_r} rowsum
  block_mm(C, Dv, Dk, [&](int i, int kk) { return Qc[i * Dk + kk]; },
           [&](int kk, int j) { return S[(size_t)kk * Dv + j]; },
           [&](int i, int j, float acc) { Tmp[i * Dv + j] = acc * dO_at(i, j); });
  __syncthreads();
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float rs = 0.f;
    for (int j = 0; j < Dv; ++j) rs += Tmp[t * Dv + j];
    dG[t] += p.scale * ev[t] * rs;
  }
  __syncthreads();
  // Tmp = (K dS) * Delta -> dc_s; <S, dS>
  block_mm(C, Dv, Dk, [&](int i, int kk) { return Kc[i * Dk + kk]; },
           [&](int kk, int j) { return dSg[(size_t)kk * Dv + j]; },
           [&](int i, int j, float acc) { Tmp[i * Dv + j] = acc * Dl[i * Dv + j]; });
  float sds = 0.f;
  for (size_t e = threadIdx.x; e < SZ; e += kThreads) sds = fmaf(S[e], dSg[e], sds);
  sds = warp_sum(sds);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sds;
  __syncthreads();
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float dc = 0.f;
    for (int j = 0; j < Dv; ++j) dc += Tmp[t * Dv + j];
    X[t] = dc * cv[t];   // X used as a [C] scratch here
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f, sum_dc = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
    for (int t = 0; t < C; ++t) sum_dc += X[t];
    dG[len - 1] += expf(gv[len - 1]) * tot + sum_dc;
  }
  __syncthreads();
  if (threadIdx.x < C) dG[threadIdx.x] -= X[threadIdx.x];
  // dW = -dDelta S^T
  block_mm(C, Dk, Dv, [&](int i, int j) { return dDc[i * Dv + j]; },
           [&](int j, int kk) { return S[(size_t)kk * Dv + j]; },
           [&](int i, int kk, float acc) { dW[i * Dk + kk] = -acc; });
  __syncthreads();
  // dT = dDelta (b V)^T + dW (b e^G K)^T, columns of valid rows only
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int r = idx / C, s = idx % C;
    float a1 = 0.f, a2 = 0.f;
    if (s < len) {
      for (int j = 0; j < Dv; ++j) a1 = fmaf(dDc[r * Dv + j], V_at(s, j), a1);
      for (int kk = 0; kk < Dk; ++kk) a2 = fmaf(dW[r * Dk + kk], Kc[s * Dk + kk], a2);
    }
    dT[idx] = bv[s] * a1 + bv[s] * ev[s] * a2;
  }
  // dBv = T^T dDelta: dv = b dBv, db += rowsum(dBv * V)
  T* dvc = (T*)p.dv + t0 * p.dv_ld + (int64_t)h * Dv;
  block_mm(C, Dv, C, [&](int s, int r) { return Tc[r * C + s]; },
           [&](int r, int j) { return dDc[r * Dv + j]; },
           [&](int s, int j, float acc) {
             Tmp[s * Dv + j] = acc * V_at(s, j);
             if (s < len) stf(dvc + (int64_t)s * p.dv_ld + j, bv[s] * acc);
           });
  __syncthreads();
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float rs = 0.f;
    for (int j = 0; j < Dv; ++j) rs += Tmp[t * Dv + j];
    db[t] += rs;
  }
  __syncthreads();
  // dBk = T^T dW: dK_hat += b e^G dBk; t = rowsum(dBk * K): db += e^G t, dG += b e^G t
  block_mm(C, Dk, C, [&](int s, int r) { return Tc[r * C + s]; },
           [&](int r, int kk) { return dW[r * Dk + kk]; },
           [&](int s, int kk, float acc) {
             dKh[s * Dk + kk] += bv[s] * ev[s] * acc;
             Tmp[s * Dk + kk] = acc * Kc[s * Dk + kk];
           });
  __syncthreads();
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float rs = 0.f;
    for (int kk = 0; kk < Dk; ++kk) rs += Tmp[t * Dk + kk];
    db[t] += ev[t] * rs;
    dG[t] += bv[t] * ev[t] * rs;
  }
  // dA = -(T^T dT T^T), strictly lower.  X = T^T dT first.
  block_mm(C, C, C, [&](int i, int r) { return Tc[r * C + i]; },
           [&](int r, int j) { return dT[r * C + j]; },
           [&](int i, int j, float acc) { X[i * C + j] = acc; });
  __syncthreads();
  block_mm(C, C, C, [&](int i, int r) { return X[i * C + r]; },
           [&](int r, int j) { return Tc[j * C + r]; },
           [&](int i, int j, float acc) { dP[i * C + j] = (j < i) ? -acc : 0.f; });
  __syncthreads();
  // A_rs = b_r E_rs KK_rs: db_r += sum_s dA E KK; Y = dA * A: dG_r += rowsum, dG_s -= colsum
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    float rdb = 0.f, ry = 0.f, cy = 0.f;
    for (int s = 0; s < t; ++s) {
      const float q = dP[t * C + s] * E[t * C + s] * KK[t * C + s];
      rdb += q;
      ry += q * bv[t];
    }
    for (int r = t + 1; r < C; ++r) cy += dP[r * C + t] * E[r * C + t] * KK[r * C + t] * bv[r];
    db[t] += rdb;
    dG[t] += ry - cy;
  }
  // H = dA * b_r E: dK_hat += H K + H^T K
  block_mm(C, Dk, C, [&](int s, int r) {
             return dP[s * C + r] * bv[s] * E[s * C + r] + dP[r * C + s] * bv[r] * E[r * C + s];
           },
           [&](int r, int kk) { return Kc[r * Dk + kk]; },
           [&](int s, int kk, float acc) { dKh[s * Dk + kk] += acc; });
  __syncthreads();
  // Gate and sigmoid epilogues (gdn_backward steps 4e, 4h): dl = reverse cumsum of dG.
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int t = C - 1; t >= 0; --t) {
      run += (t < len) ? dG[t] : 0.f;
      X[t] = run;
    }
  }
  __syncthreads();
  float pa = 0.f, pd = 0.f;
  if (threadIdx.x < C) {
    const int t = threadIdx.x;
    if (t < len) {
      const float x = p.alpha[(t0 + t) * p.alpha_ld + h] + p.dt_bias[h];
      const float ea = expf(p.a_log[h]);
      const float l = -ea * softplus_f(x);
      const float dl = X[t];
      const float da = dl * (-ea) * sigmoid_f(x);
      p.dalpha[(t0 + t) * p.dalpha_ld + h] = da;
      p.dbeta[(t0 + t) * p.dbeta_ld + h] = db[t] * bv[t] * (1.f - bv[t]);
      pa = dl * l;
      pd = da;
    }
  }
  pa = warp_sum(pa);
  pd = warp_sum(pd);
  __syncthreads();
  if (threadIdx.x < C && (threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = pa;
    red[2 + (threadIdx.x >> 5)] = pd;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.pa[ch] = red[0] + red[1];
    p.pd[ch] = red[2] + red[3];
  }
}

// dq, dk of each key head: sum of the value heads' dQ_hat / dK_hat partials in
// ascending head order, then the L2-norm backward (gdn_backward step 4f):
// dx = (dx_hat - x_hat (x_hat . dx_hat)) / sqrt(|x|^2 + 1e-6).
template <typename T>
__global__ void __launch_bounds__(kThreads) k_bwd_qk(Params p) {
  if (kept_operands_missing(p)) return;
  const int c = blockIdx.x, kh = blockIdx.y;
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  const int Dk = p.Dk, C = kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t ck = ((size_t)c * p.Hk + kh) * C;
  for (int row = warp; row < 2 * len; row += kThreads / 32) {
    const bool isk = row >= len;
    const int r = isk ? row - len : row;
    const float* xh = (isk ? p.Kn : p.Qn) + (ck + r) * Dk;
    const float* part = isk ? p.dKh : p.dQh;
    float g[4];
    float dot = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = lane + 32 * u;
      g[u] = 0.f;
      if (i < Dk) {
        for (int hh = 0; hh < p.r; ++hh)
          g[u] += part[(((size_t)c * p.Hv + value_head(p, kh, hh)) * C + r) * Dk + i];
        dot = fmaf(g[u], xh[i], dot);
      }
    }
    dot = warp_sum(dot);
    const float nrm = (isk ? p.nk : p.nq)[ck + r];
    T* dst = (T*)(isk ? p.dk : p.dq) + (t0 + r) * (isk ? p.dk_ld : p.dq_ld) + (int64_t)kh * Dk;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = lane + 32 * u;
      if (i < Dk) stf(dst + i, (g[u] - xh[i] * dot) / nrm);
    }
  }
}

__global__ void k_bwd_gates(Params p) {
  if (kept_operands_missing(p)) return;
  for (int h = threadIdx.x; h < p.Hv; h += blockDim.x) {
    float a = 0.f, d = 0.f;
    for (int c = 0; c < p.NC; ++c) {
      a += p.pa[(size_t)c * p.Hv + h];
      d += p.pd[(size_t)c * p.Hv + h];
    }
    p.da_log[h] = a;
    p.ddt_bias[h] = d;
  }
}

template <typename T>
static cudaError_t launch_backward_t(const Params& p, cudaStream_t st) {
  const int C = kChunk;
  const int DVS = p.Dv < 32 ? p.Dv : 32;
  size_t smem = sizeof(float) * ((size_t)p.Dk * DVS + (size_t)C * DVS + C * C + 3 * C);
  cudaFuncSetAttribute(k_bwd_state<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_BWD_STATE);
  k_bwd_state<T><<<dim3(p.n_seqs, p.Hv, p.Dv / DVS), kThreads, smem, st>>>(p, DVS);
  profile_post(st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int Dm = p.Dk > p.Dv ? p.Dk : p.Dv;
  smem = sizeof(float) * ((size_t)C * p.Dv + (size_t)C * p.Dk + (size_t)C * Dm + 6 * C * C +
                          6 * C + kThreads / 32);
  cudaFuncSetAttribute(k_bwd_grads<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_BWD_GRADS);
  k_bwd_grads<T><<<dim3(p.NC, p.Hv), kThreads, smem, st>>>(p);
  profile_post(st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  profile_pre(st, KID_BWD_QK);
  k_bwd_qk<T><<<dim3(p.NC, p.Hk), kThreads, 0, st>>>(p);
  profile_post(st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  profile_pre(st, KID_BWD_GATES);
  k_bwd_gates<<<1, kThreads, 0, st>>>(p);
  profile_post(st);
  return cudaGetLastError();
}

cudaError_t launch_backward(const Params& p, const TmaMaps* maps, cudaStream_t st) {
  const bool bf16 = maps != nullptr;
  if (p.NC == 0) {
    // No tokens: gradients of the per-head parameters are zero, dS_0 = dS_T.
    profile_pre(st, KID_BWD_GATES);
    k_bwd_gates<<<1, kThreads, 0, st>>>(p);
    profile_post(st);
    return cudaGetLastError();
  }
  if (bf16) {
    // bf16 inputs: tensor-core preparation, reverse state walk and gradients
    if (!p.reuse) {
      cudaError_t e = launch_prep_tc(p, *maps, true, st);
      if (e != cudaSuccess) return e;
    }
    return launch_bwd_tc(p, *maps, st);
  }
  if (!p.reuse) {
    cudaError_t e = launch_prep(p, true, st);
    if (e != cudaSuccess) return e;
  }
  return launch_backward_t<float>(p, st);
}

}  // namespace gdn
