// gdn_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously correct CPU statement of the Gated DeltaNet
// recurrence, forward and reverse-mode backward, token by token, in f64.  It
// shares no code with the CUDA path: only tests/, the smoke check and the CPU
// baseline leg of bench.py may load it.
//
// What it follows (lattice-inference 0.6.0, src/attention/gdn_backward.rs, as
// shown on docs.rs):
//   * module header "Forward recap": per value head h the key head is h / ratio
//     (head_map 0); with head_map 1 it is h % Hk, the broadcast of the ggml page's
//     op ("modulo convention");
//     g = exp(-exp(a_log[h]) * softplus(alpha + dt_bias[h])); retrieval from the
//     pre-decayed state kv_mem = S_{t-1}^T k_hat; delta = (v - g kv_mem) beta;
//     S_t = g S_{t-1} + k_hat delta^T; o_t = scale S_t^T q_hat, scale = 1/sqrt(Dk).
//   * gdn_forward_save, "L2-normalize q, k": q_hat = q / sqrt(|q|^2 + 1e-6) (the
//     eps-stabilised denominator is the one used; the max-clamped norm is only
//     saved there).
//   * gdn_backward, section 4 "Per value-head recurrence backward", steps 4a-4h
//     (o backward, state-update backward, delta backward, retrieval backward,
//     gate backward, L2-norm backward, accumulation over the value heads that
//     share a key head, sigmoid backward).  d_beta is formed without dividing by
//     beta, as step 4c there does.
// Readings where the page is silent:
//   * S_0 and dS_T are inputs (zero when absent); dS_0 is returned.
//   * d a_log[h] = sum over every token of every sequence of dl * l (dl/d a_log
//     = l because l = -exp(a_log) softplus(x)); d dt_bias[h] = sum of d alpha.
//   * softplus(x) = max(x, 0) + log1p(exp(-|x|)), the exact log(1 + e^x).
//   * varlen: each sequence of cu_seqlens starts from its own S_0[n].
//
// Memory: the backward keeps a state checkpoint every `segment` tokens and
// recomputes the states inside one segment before walking it in reverse.
// Work is split over (sequence, key head) units on std::threads; the only
// cross-unit sums (d a_log, d dt_bias) are reduced in sequence order after
// the threads join, so results do not depend on the thread count.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  int32_t Hk, Hv, Dk, Dv;
  int32_t n_seqs;
  int64_t total_tokens;
  double scale;       // <= 0 selects 1/sqrt(Dk)
  int32_t n_threads;  // <= 0 selects std::thread::hardware_concurrency()
  int32_t segment;    // backward checkpoint interval in tokens; <= 0 selects 64
  int32_t head_map;   // 0: key head of value head h is h / (Hv/Hk); 1: h % Hk
} gdn_oracle_shape;

typedef struct {
  const double* q;        int64_t q_ld;      // [T, q_ld], key head kh at column kh*Dk
  const double* k;        int64_t k_ld;      // [T, k_ld], key head kh at column kh*Dk
  const double* v;        int64_t v_ld;      // [T, v_ld], value head h at column h*Dv
  const double* alpha;    int64_t alpha_ld;  // [T, alpha_ld], column h
  const double* beta_raw; int64_t beta_ld;   // [T, beta_ld], column h
  const double* a_log;                       // [Hv]
  const double* dt_bias;                     // [Hv]
  const int32_t* cu_seqlens;                 // [n_seqs + 1]
  const double* S0;                          // [n_seqs, Hv, Dk, Dv] or NULL (zero)
} gdn_oracle_inputs;

int gdn_oracle_forward(const gdn_oracle_shape* shape, const gdn_oracle_inputs* in,
                       double* o, int64_t o_ld, double* S_T);
// As gdn_oracle_forward, and also writes the state at the start of every
// `chunk`-token chunk of every sequence: chunk_states[c, Hv, Dk, Dv] with the
// chunks of sequence n numbered from chunk_offsets[n] (chunks never span two
// sequences; the last chunk of a sequence may be short).
int gdn_oracle_forward_states(const gdn_oracle_shape* shape, const gdn_oracle_inputs* in,
                              double* o, int64_t o_ld, double* S_T, int32_t chunk,
                              const int32_t* chunk_offsets, double* chunk_states);
int gdn_oracle_backward(const gdn_oracle_shape* shape, const gdn_oracle_inputs* in,
                        const double* dO, int64_t dO_ld, const double* dS_T,
                        double* dq, int64_t dq_ld, double* dk, int64_t dk_ld,
                        double* dv, int64_t dv_ld, double* dalpha, int64_t dalpha_ld,
                        double* dbeta_raw, int64_t dbeta_ld, double* da_log,
                        double* ddt_bias, double* dS0);
int gdn_oracle_hardware_threads(void);

}  // extern "C"

namespace {

double softplus(double x) { return std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x))); }
double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

struct Dims {
  int Hk, Hv, Dk, Dv, r, head_map;
  double scale;
  int64_t DkDv() const { return (int64_t)Dk * Dv; }
  // value head number hh (0 <= hh < r) of key head kh
  int vh(int kh, int hh) const { return head_map ? kh + hh * Hk : kh * r + hh; }
};

// Gate quantities of value head h at token t.
struct Gate {
  double b;  // beta = sigmoid(beta_raw)
  double x;  // alpha + dt_bias
  double l;  // log g = -exp(a_log) softplus(x)
  double g;  // decay
};

Gate gate_at(const gdn_oracle_inputs& in, int64_t t, int h) {
  Gate G;
  G.b = sigmoid(in.beta_raw[t * in.beta_ld + h]);
  G.x = in.alpha[t * in.alpha_ld + h] + in.dt_bias[h];
  G.l = -std::exp(in.a_log[h]) * softplus(G.x);
  G.g = std::exp(G.l);
  return G;
}

// xhat = x / sqrt(|x|^2 + 1e-6); returns the denominator.
double l2_normalise(const double* x, int D, double* xhat) {
  double ss = 0.0;
  for (int i = 0; i < D; ++i) ss += x[i] * x[i];
  const double n = std::sqrt(ss + 1e-6);
  for (int i = 0; i < D; ++i) xhat[i] = x[i] / n;
  return n;
}

// One forward token step of one value head.  S is Dk x Dv row-major and is
// updated in place; kv (retrieval) and delta are returned for the caller.
void token_step(const Dims& d, double* S, const double* khat, const double* v, const Gate& G,
                double* kv, double* delta) {
  for (int j = 0; j < d.Dv; ++j) kv[j] = 0.0;
  for (int i = 0; i < d.Dk; ++i)
    for (int j = 0; j < d.Dv; ++j) kv[j] += S[(int64_t)i * d.Dv + j] * khat[i];
  for (int j = 0; j < d.Dv; ++j) delta[j] = G.b * (v[j] - G.g * kv[j]);
  for (int i = 0; i < d.Dk; ++i)
    for (int j = 0; j < d.Dv; ++j)
      S[(int64_t)i * d.Dv + j] = G.g * S[(int64_t)i * d.Dv + j] + khat[i] * delta[j];
}

template <typename F>
void run_units(int n_units, int n_threads, F&& fn) {
  if (n_threads <= 0) n_threads = (int)std::max(1u, std::thread::hardware_concurrency());
  n_threads = std::max(1, std::min(n_threads, n_units));
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (;;) {
      const int u = next.fetch_add(1);
      if (u >= n_units) return;
      fn(u);
    }
  };
  if (n_threads == 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int i = 0; i < n_threads; ++i) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

int check_shape(const gdn_oracle_shape* s, const gdn_oracle_inputs* in, Dims* d) {
  if (!s || !in) return -1;
  if (s->Hk <= 0 || s->Hv <= 0 || s->Dk <= 0 || s->Dv <= 0 || s->n_seqs < 0) return -1;
  if (s->Hv % s->Hk != 0) return -1;
  if (!in->cu_seqlens) return -1;
  if (in->cu_seqlens[0] != 0 || in->cu_seqlens[s->n_seqs] != s->total_tokens) return -1;
  for (int n = 0; n < s->n_seqs; ++n)
    if (in->cu_seqlens[n + 1] < in->cu_seqlens[n]) return -1;
  d->Hk = s->Hk;
  d->Hv = s->Hv;
  d->Dk = s->Dk;
  d->Dv = s->Dv;
  d->r = s->Hv / s->Hk;
  if (s->head_map != 0 && s->head_map != 1) return -1;
  d->head_map = s->head_map;
  d->scale = s->scale > 0.0 ? s->scale : 1.0 / std::sqrt((double)s->Dk);
  return 0;
}

}  // namespace

extern "C" int gdn_oracle_hardware_threads(void) {
  return (int)std::max(1u, std::thread::hardware_concurrency());
}

extern "C" int gdn_oracle_forward(const gdn_oracle_shape* shape, const gdn_oracle_inputs* inp,
                                  double* o, int64_t o_ld, double* S_T) {
  return gdn_oracle_forward_states(shape, inp, o, o_ld, S_T, 0, nullptr, nullptr);
}

extern "C" int gdn_oracle_forward_states(const gdn_oracle_shape* shape,
                                         const gdn_oracle_inputs* inp, double* o, int64_t o_ld,
                                         double* S_T, int32_t chunk,
                                         const int32_t* chunk_offsets, double* chunk_states) {
  Dims d;
  if (check_shape(shape, inp, &d) != 0 || !o) return -1;
  if (chunk_states && (chunk <= 0 || !chunk_offsets)) return -1;
  const gdn_oracle_inputs& in = *inp;
  const int n_units = shape->n_seqs * d.Hk;
  run_units(n_units, shape->n_threads, [&](int u) {
    const int n = u / d.Hk, kh = u % d.Hk;
    const int64_t t0 = in.cu_seqlens[n], t1 = in.cu_seqlens[n + 1];
    std::vector<double> S((size_t)d.r * d.DkDv(), 0.0);
    if (in.S0)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(&S[(size_t)hh * d.DkDv()], in.S0 + ((int64_t)n * d.Hv + d.vh(kh, hh)) * d.DkDv(),
                    sizeof(double) * d.DkDv());
    std::vector<double> qh(d.Dk), kh_(d.Dk), kv(d.Dv), delta(d.Dv);
    for (int64_t t = t0; t < t1; ++t) {
      if (chunk_states && (t - t0) % chunk == 0) {
        const int64_t c = chunk_offsets[n] + (t - t0) / chunk;
        for (int hh = 0; hh < d.r; ++hh)
          std::memcpy(chunk_states + (c * d.Hv + d.vh(kh, hh)) * d.DkDv(), &S[(size_t)hh * d.DkDv()],
                      sizeof(double) * d.DkDv());
      }
      l2_normalise(in.q + t * in.q_ld + (int64_t)kh * d.Dk, d.Dk, qh.data());
      l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, kh_.data());
      for (int hh = 0; hh < d.r; ++hh) {
        const int h = d.vh(kh, hh);
        double* Sh = &S[(size_t)hh * d.DkDv()];
        const Gate G = gate_at(in, t, h);
        token_step(d, Sh, kh_.data(), in.v + t * in.v_ld + (int64_t)h * d.Dv, G, kv.data(),
                   delta.data());
        double* orow = o + t * o_ld + (int64_t)h * d.Dv;
        for (int j = 0; j < d.Dv; ++j) orow[j] = 0.0;
        for (int i = 0; i < d.Dk; ++i)
          for (int j = 0; j < d.Dv; ++j) orow[j] += Sh[(int64_t)i * d.Dv + j] * qh[i];
        for (int j = 0; j < d.Dv; ++j) orow[j] *= d.scale;
      }
    }
    if (S_T)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(S_T + ((int64_t)n * d.Hv + d.vh(kh, hh)) * d.DkDv(), &S[(size_t)hh * d.DkDv()],
                    sizeof(double) * d.DkDv());
  });
  return 0;
}

extern "C" int gdn_oracle_backward(const gdn_oracle_shape* shape, const gdn_oracle_inputs* inp,
                                   const double* dO, int64_t dO_ld, const double* dS_T,
                                   double* dq, int64_t dq_ld, double* dk, int64_t dk_ld,
                                   double* dv, int64_t dv_ld, double* dalpha, int64_t dalpha_ld,
                                   double* dbeta_raw, int64_t dbeta_ld, double* da_log,
                                   double* ddt_bias, double* dS0) {
  Dims d;
  if (check_shape(shape, inp, &d) != 0) return -1;
  if (!dO || !dq || !dk || !dv || !dalpha || !dbeta_raw || !da_log || !ddt_bias) return -1;
  const gdn_oracle_inputs& in = *inp;
  const int seg = shape->segment > 0 ? shape->segment : 64;
  const int N = shape->n_seqs;
  // Per (sequence, value head) partial sums of d a_log and d dt_bias.
  std::vector<double> pa((size_t)std::max(N, 1) * d.Hv, 0.0), pd((size_t)std::max(N, 1) * d.Hv, 0.0);
  const int n_units = N * d.Hk;
  run_units(n_units, shape->n_threads, [&](int u) {
    const int n = u / d.Hk, kh = u % d.Hk;
    const int64_t t0 = in.cu_seqlens[n], t1 = in.cu_seqlens[n + 1];
    const int64_t L = t1 - t0;
    const int64_t n_seg = (L + seg - 1) / seg;
    const size_t SZ = (size_t)d.DkDv();
    // Checkpoints: state of each value head of the group before token t0 + s*seg.
    std::vector<double> ck((size_t)std::max<int64_t>(n_seg, 1) * d.r * SZ, 0.0);
    std::vector<double> S((size_t)d.r * SZ, 0.0);
    if (in.S0)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(&S[hh * SZ], in.S0 + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ, sizeof(double) * SZ);
    std::vector<double> qh(d.Dk), khat(d.Dk), kv(d.Dv), delta(d.Dv);
    for (int64_t t = t0; t < t1; ++t) {
      if ((t - t0) % seg == 0)
        std::memcpy(&ck[(size_t)((t - t0) / seg) * d.r * SZ], S.data(), sizeof(double) * d.r * SZ);
      l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
      for (int hh = 0; hh < d.r; ++hh) {
        const int h = d.vh(kh, hh);
        token_step(d, &S[hh * SZ], khat.data(), in.v + t * in.v_ld + (int64_t)h * d.Dv,
                   gate_at(in, t, h), kv.data(), delta.data());
      }
    }
    // Adjoint of the state, one per value head of the group.
    std::vector<double> dS((size_t)d.r * SZ, 0.0);
    if (dS_T)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(&dS[hh * SZ], dS_T + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ, sizeof(double) * SZ);
    // States before each token of the current segment (plus the one after its end).
    std::vector<double> Sbuf((size_t)(seg + 1) * d.r * SZ);
    std::vector<double> S_t(SZ), dqh(d.Dk), dkh(d.Dk), ddelta(d.Dv), dkv(d.Dv);
    std::vector<double> dq_acc(d.Dk), dk_acc(d.Dk);
    for (int64_t s = n_seg - 1; s >= 0; --s) {
      const int64_t ta = t0 + s * seg, tb = std::min<int64_t>(ta + seg, t1);
      std::memcpy(&Sbuf[0], &ck[(size_t)s * d.r * SZ], sizeof(double) * d.r * SZ);
      for (int64_t t = ta; t < tb; ++t) {
        l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
        double* nxt = &Sbuf[(size_t)(t - ta + 1) * d.r * SZ];
        std::memcpy(nxt, &Sbuf[(size_t)(t - ta) * d.r * SZ], sizeof(double) * d.r * SZ);
        for (int hh = 0; hh < d.r; ++hh) {
          const int h = d.vh(kh, hh);
          token_step(d, nxt + hh * SZ, khat.data(), in.v + t * in.v_ld + (int64_t)h * d.Dv,
                     gate_at(in, t, h), kv.data(), delta.data());
        }
      }
      for (int64_t t = tb - 1; t >= ta; --t) {
        const double nq = l2_normalise(in.q + t * in.q_ld + (int64_t)kh * d.Dk, d.Dk, qh.data());
        const double nk = l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
        std::fill(dq_acc.begin(), dq_acc.end(), 0.0);
        std::fill(dk_acc.begin(), dk_acc.end(), 0.0);
        for (int hh = 0; hh < d.r; ++hh) {
          const int h = d.vh(kh, hh);
          const double* S_prev = &Sbuf[(size_t)(t - ta) * d.r * SZ + hh * SZ];
          const double* vrow = in.v + t * in.v_ld + (int64_t)h * d.Dv;
          const double* dOrow = dO + t * dO_ld + (int64_t)h * d.Dv;
          double* dSh = &dS[hh * SZ];
          const Gate G = gate_at(in, t, h);
          // Recompute this token's forward quantities from the state before it.
          std::memcpy(S_t.data(), S_prev, sizeof(double) * SZ);
          token_step(d, S_t.data(), khat.data(), vrow, G, kv.data(), delta.data());
          // 4a: o = scale S_t^T q_hat.
          for (int i = 0; i < d.Dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d.Dv; ++j) {
              dSh[(int64_t)i * d.Dv + j] += d.scale * qh[i] * dOrow[j];
              acc += S_t[(int64_t)i * d.Dv + j] * dOrow[j];
            }
            dqh[i] = d.scale * acc;
          }
          // 4b: S_t = g S_prev + k_hat delta^T.
          double dg = 0.0;
          std::fill(dkh.begin(), dkh.end(), 0.0);
          std::fill(ddelta.begin(), ddelta.end(), 0.0);
          for (int i = 0; i < d.Dk; ++i)
            for (int j = 0; j < d.Dv; ++j) {
              const double ds = dSh[(int64_t)i * d.Dv + j];
              dg += S_prev[(int64_t)i * d.Dv + j] * ds;
              dkh[i] += ds * delta[j];
              ddelta[j] += ds * khat[i];
            }
          for (size_t e = 0; e < SZ; ++e) dSh[e] *= G.g;
          // 4c: delta = beta (v - g kv).
          double db = 0.0;
          for (int j = 0; j < d.Dv; ++j) {
            dv[t * dv_ld + (int64_t)h * d.Dv + j] = G.b * ddelta[j];
            dkv[j] = -G.g * G.b * ddelta[j];
            dg += -kv[j] * G.b * ddelta[j];
            db += (vrow[j] - G.g * kv[j]) * ddelta[j];
          }
          // 4d: kv = S_prev^T k_hat.
          for (int i = 0; i < d.Dk; ++i)
            for (int j = 0; j < d.Dv; ++j) {
              dSh[(int64_t)i * d.Dv + j] += khat[i] * dkv[j];
              dkh[i] += S_prev[(int64_t)i * d.Dv + j] * dkv[j];
            }
          // 4e: g = exp(l), l = -exp(a_log) softplus(x), softplus' = sigmoid.
          const double dl = dg * G.g;
          const double da = dl * (-std::exp(in.a_log[h])) * sigmoid(G.x);
          dalpha[t * dalpha_ld + h] = da;
          pa[(size_t)n * d.Hv + h] += dl * G.l;
          pd[(size_t)n * d.Hv + h] += da;
          // 4f + 4g: L2-norm backward, summed over the value heads of this key head.
          double dot_q = 0.0, dot_k = 0.0;
          for (int i = 0; i < d.Dk; ++i) {
            dot_q += dqh[i] * qh[i];
            dot_k += dkh[i] * khat[i];
          }
          for (int i = 0; i < d.Dk; ++i) {
            dq_acc[i] += (dqh[i] - qh[i] * dot_q) / nq;
            dk_acc[i] += (dkh[i] - khat[i] * dot_k) / nk;
          }
          // 4h: beta = sigmoid(beta_raw).
          dbeta_raw[t * dbeta_ld + h] = db * G.b * (1.0 - G.b);
        }
        for (int i = 0; i < d.Dk; ++i) {
          dq[t * dq_ld + (int64_t)kh * d.Dk + i] = dq_acc[i];
          dk[t * dk_ld + (int64_t)kh * d.Dk + i] = dk_acc[i];
        }
      }
    }
    if (dS0)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(dS0 + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ, &dS[hh * SZ], sizeof(double) * SZ);
  });
  for (int h = 0; h < d.Hv; ++h) {
    double a = 0.0, b = 0.0;
    for (int n = 0; n < N; ++n) {
      a += pa[(size_t)n * d.Hv + h];
      b += pd[(size_t)n * d.Hv + h];
    }
    da_log[h] = a;
    ddt_bias[h] = b;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// The layer steps on either side of the recurrence, from the forward of lattice-inference
// 0.6.0, src/attention/gdn_backward.rs (its "Causal conv1d + SiLU" and "Gated RMSNorm +
// output projection" steps) and its backward (sections 2 and 5), in f64 with plain loops.  Readings where the page is silent:
//   * the conv's rolling buffer starts at zero at every sequence start (varlen);
//   * the weight gradients dw (conv) and dgamma (norm), which the page does not form
//     (its base weights are frozen), are the sums over every token of the products
//     the forward multiplies the weights into;
//   * rms_eps is an argument.

namespace {
double silu(double x) { return x / (1.0 + std::exp(-x)); }
double silu_grad(double x) {  // d/dx x sigmoid(x) = sigmoid(x) (1 + x (1 - sigmoid(x)))
  const double s = 1.0 / (1.0 + std::exp(-x));
  return s * (1.0 + x * (1.0 - s));
}
// Pre-activation of channel ch at token t (sequence start t_start): the page's
// sum_pre = sum_tb buf[ch,tb] w[ch*K + tb] + x[t][ch] w[ch*K + K-1], buf[ch,tb] the
// input K-1-tb tokens back (zero before the sequence start).
double conv_pre(const double* x, int64_t x_ld, const double* w, int K, int ch, int64_t t,
                int64_t t_start) {
  double s = 0.0;
  for (int j = 0; j < K; ++j) {
    const int64_t src = t - (K - 1 - j);
    if (src >= t_start) s += x[src * x_ld + ch] * w[(int64_t)ch * K + j];
  }
  return s;
}
bool check_cu(int32_t n_seqs, const int32_t* cu, int64_t T) {
  if (!cu || n_seqs < 0 || cu[0] != 0 || cu[n_seqs] != T) return false;
  for (int n = 0; n < n_seqs; ++n)
    if (cu[n + 1] < cu[n]) return false;
  return true;
}
}  // namespace

extern "C" int gdn_oracle_conv1d_silu_forward(int64_t T, int32_t C, int32_t K, int32_t n_seqs,
                                               const int32_t* cu, const double* x, int64_t x_ld,
                                               const double* w, double* y, int64_t y_ld) {
  if (C <= 0 || K <= 0 || !x || !w || !y || !check_cu(n_seqs, cu, T)) return -1;
  for (int n = 0; n < n_seqs; ++n)
    for (int64_t t = cu[n]; t < cu[n + 1]; ++t)
      for (int ch = 0; ch < C; ++ch)
        y[t * y_ld + ch] = silu(conv_pre(x, x_ld, w, K, ch, t, cu[n]));
  return 0;
}

// Backward (the page's section 5): d_sum = dy * SiLU'(sum_pre); the input K-1-j tokens
// before an output gets d_sum * w[ch*K + j]; dw[ch*K + j] sums d_sum times that input.
extern "C" int gdn_oracle_conv1d_silu_backward(int64_t T, int32_t C, int32_t K, int32_t n_seqs,
                                                const int32_t* cu, const double* x, int64_t x_ld,
                                                const double* w, const double* dy, int64_t dy_ld,
                                                double* dx, int64_t dx_ld, double* dw) {
  if (C <= 0 || K <= 0 || !x || !w || !dy || !dx || !check_cu(n_seqs, cu, T)) return -1;
  for (int64_t t = 0; t < T; ++t)
    for (int ch = 0; ch < C; ++ch) dx[t * dx_ld + ch] = 0.0;
  if (dw)
    for (int64_t i = 0; i < (int64_t)C * K; ++i) dw[i] = 0.0;
  for (int n = 0; n < n_seqs; ++n)
    for (int64_t t = cu[n]; t < cu[n + 1]; ++t)
      for (int ch = 0; ch < C; ++ch) {
        const double d_sum = dy[t * dy_ld + ch] * silu_grad(conv_pre(x, x_ld, w, K, ch, t, cu[n]));
        for (int j = 0; j < K; ++j) {
          const int64_t src = t - (K - 1 - j);
          if (src < cu[n]) continue;
          dx[src * dx_ld + ch] += d_sum * w[(int64_t)ch * K + j];
          if (dw) dw[(int64_t)ch * K + j] += d_sum * x[src * x_ld + ch];
        }
      }
  return 0;
}

// Gated RMSNorm of every (token, value head): rms = sqrt(mean_j o_j^2 + eps),
// y_j = (o_j / rms) gamma_j SiLU(z_j), gamma shared by the heads.
extern "C" int gdn_oracle_gated_rmsnorm_forward(int64_t T, int32_t H, int32_t D, double eps,
                                                 const double* o, int64_t o_ld, const double* z,
                                                 int64_t z_ld, const double* gamma, double* y,
                                                 int64_t y_ld) {
  if (T < 0 || H <= 0 || D <= 0 || !o || !z || !gamma || !y) return -1;
  for (int64_t t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      const double* oh = o + t * o_ld + (int64_t)h * D;
      const double* zh = z + t * z_ld + (int64_t)h * D;
      double ss = 0.0;
      for (int j = 0; j < D; ++j) ss += oh[j] * oh[j];
      const double rms = std::sqrt(ss / D + eps);
      for (int j = 0; j < D; ++j) y[t * y_ld + (int64_t)h * D + j] = oh[j] / rms * gamma[j] * silu(zh[j]);
    }
  return 0;
}

// Backward (the page's section 2): d_xnorm = dy gamma SiLU(z); dz = dy gamma x_norm
// SiLU'(z); do = d_xnorm / rms - o (sum_k d_xnorm_k o_k) / (rms^3 D); dgamma sums
// dy x_norm SiLU(z) over every token and head.
extern "C" int gdn_oracle_gated_rmsnorm_backward(int64_t T, int32_t H, int32_t D, double eps,
                                                  const double* o, int64_t o_ld, const double* z,
                                                  int64_t z_ld, const double* gamma,
                                                  const double* dy, int64_t dy_ld, double* d_o,
                                                  int64_t do_ld, double* dz, int64_t dz_ld,
                                                  double* dgamma) {
  if (T < 0 || H <= 0 || D <= 0 || !o || !z || !gamma || !dy || !d_o || !dz) return -1;
  if (dgamma)
    for (int j = 0; j < D; ++j) dgamma[j] = 0.0;
  std::vector<double> dxn(D);
  for (int64_t t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      const double* oh = o + t * o_ld + (int64_t)h * D;
      const double* zh = z + t * z_ld + (int64_t)h * D;
      const double* dg = dy + t * dy_ld + (int64_t)h * D;
      double ss = 0.0;
      for (int j = 0; j < D; ++j) ss += oh[j] * oh[j];
      const double rms = std::sqrt(ss / D + eps);
      double dot = 0.0;
      for (int j = 0; j < D; ++j) {
        const double xn = oh[j] / rms;
        dxn[j] = dg[j] * gamma[j] * silu(zh[j]);
        dz[t * dz_ld + (int64_t)h * D + j] = dg[j] * gamma[j] * xn * silu_grad(zh[j]);
        if (dgamma) dgamma[j] += dg[j] * xn * silu(zh[j]);
        dot += dxn[j] * oh[j];
      }
      for (int j = 0; j < D; ++j)
        d_o[t * do_ld + (int64_t)h * D + j] = dxn[j] / rms - oh[j] * dot / (rms * rms * rms * D);
    }
  return 0;
}

// ---------------------------------------------------------------------------
// The linear part of a sequence's state map, for splitting one sequence over several
// workers (context parallelism).  The token update of the forward recap above rewrites as
//   S_t = g_t (I - beta_t k_hat_t k_hat_t^T) S_{t-1} + beta_t k_hat_t v_t^T,
// so a sequence maps its start state affinely, S_T = Phi S_0 + R, with
//   Phi = A_L ... A_2 A_1,  A_t = g_t (I - beta_t k_hat_t k_hat_t^T)   (Dk x Dk),
// and R the final state from S_0 = 0.  Phi is formed here by applying each A_t in turn to
// the identity; Phi[n, h] is [Dk, Dk] row-major, value head h of sequence n.
extern "C" int gdn_oracle_state_map(const gdn_oracle_shape* shape, const gdn_oracle_inputs* inp,
                                    double* Phi) {
  Dims d;
  if (check_shape(shape, inp, &d) != 0 || !Phi) return -1;
  const gdn_oracle_inputs& in = *inp;
  const int64_t DD = (int64_t)d.Dk * d.Dk;
  run_units(shape->n_seqs * d.Hv, shape->n_threads, [&](int u) {
    const int n = u / d.Hv, h = u % d.Hv;
    const int kh = d.head_map ? h % d.Hk : h / d.r;
    double* P = Phi + ((int64_t)n * d.Hv + h) * DD;
    for (int64_t i = 0; i < DD; ++i) P[i] = 0.0;
    for (int i = 0; i < d.Dk; ++i) P[(int64_t)i * d.Dk + i] = 1.0;
    std::vector<double> kh_(d.Dk), w(d.Dk);
    for (int64_t t = in.cu_seqlens[n]; t < in.cu_seqlens[n + 1]; ++t) {
      l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, kh_.data());
      const Gate G = gate_at(in, t, h);
      // P <- g (P - beta k_hat (k_hat^T P))
      for (int j = 0; j < d.Dk; ++j) w[j] = 0.0;
      for (int i = 0; i < d.Dk; ++i)
        for (int j = 0; j < d.Dk; ++j) w[j] += kh_[i] * P[(int64_t)i * d.Dk + j];
      for (int i = 0; i < d.Dk; ++i)
        for (int j = 0; j < d.Dk; ++j)
          P[(int64_t)i * d.Dk + j] = G.g * (P[(int64_t)i * d.Dk + j] - G.b * kh_[i] * w[j]);
    }
  });
  return 0;
}

// ---------------------------------------------------------------------------
// KDA variant: the recurrence with a decay gate per key channel instead of one per head
// (the dormouse "KDA attention arm" page names the module's decay parameters a_log and
// b_alpha; the recurrence itself is not printed there).  Reading: channel c of value head
// h decays by g[c] = exp(l[c]), l[c] = -exp(a_log[h]) softplus(alpha[t, h*Dk + c] +
// b_alpha[h*Dk + c]), and the forward recap's update becomes
//   S_d = diag(g) S_{t-1},  kv = S_d^T k_hat,  delta = beta (v - kv),
//   S_t = S_d + k_hat delta^T,  o_t = scale S_t^T q_hat.
// With every channel's alpha and b_alpha equal it is the scalar-gate recurrence above.
// In the input struct, alpha is [T, alpha_ld >= Hv*Dk] and dt_bias holds b_alpha [Hv*Dk].
// Plain loops per (sequence, value head); the backward keeps every state of a unit
// (small shapes only).
namespace {
void kda_gates(const gdn_oracle_inputs& in, const Dims& d, int64_t t, int h, double* g,
               double* l, double* x) {
  for (int c = 0; c < d.Dk; ++c) {
    x[c] = in.alpha[t * in.alpha_ld + (int64_t)h * d.Dk + c] + in.dt_bias[(int64_t)h * d.Dk + c];
    l[c] = -std::exp(in.a_log[h]) * softplus(x[c]);
    g[c] = std::exp(l[c]);
  }
}
// One KDA token step of one value head: S (Dk x Dv) updated in place; kv and delta out.
void kda_step(const Dims& d, double* S, const double* khat, const double* v, const double* g,
              double b, double* kv, double* delta) {
  for (int i = 0; i < d.Dk; ++i)
    for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] *= g[i];
  for (int j = 0; j < d.Dv; ++j) kv[j] = 0.0;
  for (int i = 0; i < d.Dk; ++i)
    for (int j = 0; j < d.Dv; ++j) kv[j] += S[(int64_t)i * d.Dv + j] * khat[i];
  for (int j = 0; j < d.Dv; ++j) delta[j] = b * (v[j] - kv[j]);
  for (int i = 0; i < d.Dk; ++i)
    for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] += khat[i] * delta[j];
}
}  // namespace

extern "C" int gdn_oracle_kda_forward(const gdn_oracle_shape* shape, const gdn_oracle_inputs* inp,
                                      double* o, int64_t o_ld, double* S_T) {
  Dims d;
  if (check_shape(shape, inp, &d) != 0 || !o) return -1;
  const gdn_oracle_inputs& in = *inp;
  const int64_t SZ = d.DkDv();
  run_units(shape->n_seqs * d.Hv, shape->n_threads, [&](int u) {
    const int n = u / d.Hv, h = u % d.Hv;
    const int kh = d.head_map ? h % d.Hk : h / d.r;
    std::vector<double> S(SZ, 0.0), qh(d.Dk), khat(d.Dk), kv(d.Dv), delta(d.Dv), g(d.Dk),
        l(d.Dk), x(d.Dk);
    if (in.S0) std::memcpy(S.data(), in.S0 + ((int64_t)n * d.Hv + h) * SZ, sizeof(double) * SZ);
    for (int64_t t = in.cu_seqlens[n]; t < in.cu_seqlens[n + 1]; ++t) {
      l2_normalise(in.q + t * in.q_ld + (int64_t)kh * d.Dk, d.Dk, qh.data());
      l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
      kda_gates(in, d, t, h, g.data(), l.data(), x.data());
      const double b = sigmoid(in.beta_raw[t * in.beta_ld + h]);
      kda_step(d, S.data(), khat.data(), in.v + t * in.v_ld + (int64_t)h * d.Dv, g.data(), b,
               kv.data(), delta.data());
      double* orow = o + t * o_ld + (int64_t)h * d.Dv;
      for (int j = 0; j < d.Dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d.Dk; ++i) acc += S[(int64_t)i * d.Dv + j] * qh[i];
        orow[j] = d.scale * acc;
      }
    }
    if (S_T) std::memcpy(S_T + ((int64_t)n * d.Hv + h) * SZ, S.data(), sizeof(double) * SZ);
  });
  return 0;
}

// Reverse mode of gdn_oracle_kda_forward: the adjoint steps of the scalar-gate backward
// with dg per channel, dg[c] = sum_j S_prev[c][j] dS_d[c][j].  dalpha is [T, Hv*Dk];
// ddt_bias receives d b_alpha [Hv*Dk]; both gate-parameter sums run over every token of
// every sequence, reduced in sequence order.
extern "C" int gdn_oracle_kda_backward(const gdn_oracle_shape* shape,
                                       const gdn_oracle_inputs* inp, const double* dO,
                                       int64_t dO_ld, const double* dS_T, double* dq,
                                       int64_t dq_ld, double* dk, int64_t dk_ld, double* dv,
                                       int64_t dv_ld, double* dalpha, int64_t dalpha_ld,
                                       double* dbeta_raw, int64_t dbeta_ld, double* da_log,
                                       double* db_alpha, double* dS0) {
  Dims d;
  if (check_shape(shape, inp, &d) != 0) return -1;
  if (!dO || !dq || !dk || !dv || !dalpha || !dbeta_raw || !da_log || !db_alpha) return -1;
  const gdn_oracle_inputs& in = *inp;
  const int N = shape->n_seqs;
  const int64_t SZ = d.DkDv();
  std::vector<double> pa((size_t)std::max(N, 1) * d.Hv, 0.0);
  std::vector<double> pb((size_t)std::max(N, 1) * d.Hv * d.Dk, 0.0);
  run_units(N * d.Hk, shape->n_threads, [&](int u) {
    const int n = u / d.Hk, kh = u % d.Hk;
    const int64_t t0 = in.cu_seqlens[n], t1 = in.cu_seqlens[n + 1], L = t1 - t0;
    // states before every token, per value head of the group: [L + 1][r][SZ]
    std::vector<double> Sh((size_t)(L + 1) * d.r * SZ, 0.0);
    if (in.S0)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(&Sh[hh * SZ], in.S0 + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ,
                    sizeof(double) * SZ);
    std::vector<double> qh(d.Dk), khat(d.Dk), kv(d.Dv), delta(d.Dv), g(d.Dk), l(d.Dk), x(d.Dk);
    for (int64_t t = t0; t < t1; ++t) {
      l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
      double* nxt = &Sh[(size_t)(t - t0 + 1) * d.r * SZ];
      std::memcpy(nxt, &Sh[(size_t)(t - t0) * d.r * SZ], sizeof(double) * d.r * SZ);
      for (int hh = 0; hh < d.r; ++hh) {
        const int h = d.vh(kh, hh);
        kda_gates(in, d, t, h, g.data(), l.data(), x.data());
        kda_step(d, nxt + hh * SZ, khat.data(), in.v + t * in.v_ld + (int64_t)h * d.Dv, g.data(),
                 sigmoid(in.beta_raw[t * in.beta_ld + h]), kv.data(), delta.data());
      }
    }
    std::vector<double> dS((size_t)d.r * SZ, 0.0);
    if (dS_T)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(&dS[hh * SZ], dS_T + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ,
                    sizeof(double) * SZ);
    std::vector<double> Sd(SZ), S_t(SZ), dqh(d.Dk), dkh(d.Dk), ddelta(d.Dv), dkv(d.Dv), dg(d.Dk);
    std::vector<double> dq_acc(d.Dk), dk_acc(d.Dk);
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double nq = l2_normalise(in.q + t * in.q_ld + (int64_t)kh * d.Dk, d.Dk, qh.data());
      const double nk = l2_normalise(in.k + t * in.k_ld + (int64_t)kh * d.Dk, d.Dk, khat.data());
      std::fill(dq_acc.begin(), dq_acc.end(), 0.0);
      std::fill(dk_acc.begin(), dk_acc.end(), 0.0);
      for (int hh = 0; hh < d.r; ++hh) {
        const int h = d.vh(kh, hh);
        const double* S_prev = &Sh[(size_t)(t - t0) * d.r * SZ + hh * SZ];
        const double* vrow = in.v + t * in.v_ld + (int64_t)h * d.Dv;
        const double* dOrow = dO + t * dO_ld + (int64_t)h * d.Dv;
        double* dSh = &dS[hh * SZ];
        kda_gates(in, d, t, h, g.data(), l.data(), x.data());
        const double b = sigmoid(in.beta_raw[t * in.beta_ld + h]);
        // recompute S_d, kv, delta, S_t
        for (int i = 0; i < d.Dk; ++i)
          for (int j = 0; j < d.Dv; ++j) Sd[(int64_t)i * d.Dv + j] = g[i] * S_prev[(int64_t)i * d.Dv + j];
        std::memcpy(S_t.data(), S_prev, sizeof(double) * SZ);
        kda_step(d, S_t.data(), khat.data(), vrow, g.data(), b, kv.data(), delta.data());
        // o = scale S_t^T q_hat
        for (int i = 0; i < d.Dk; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d.Dv; ++j) {
            dSh[(int64_t)i * d.Dv + j] += d.scale * qh[i] * dOrow[j];
            acc += S_t[(int64_t)i * d.Dv + j] * dOrow[j];
          }
          dqh[i] = d.scale * acc;
        }
        // S_t = S_d + k_hat delta^T  (dS_d = dS)
        std::fill(dkh.begin(), dkh.end(), 0.0);
        std::fill(ddelta.begin(), ddelta.end(), 0.0);
        for (int i = 0; i < d.Dk; ++i)
          for (int j = 0; j < d.Dv; ++j) {
            const double ds = dSh[(int64_t)i * d.Dv + j];
            dkh[i] += ds * delta[j];
            ddelta[j] += ds * khat[i];
          }
        // delta = beta (v - kv)
        double db = 0.0;
        for (int j = 0; j < d.Dv; ++j) {
          dv[t * dv_ld + (int64_t)h * d.Dv + j] = b * ddelta[j];
          dkv[j] = -b * ddelta[j];
          db += (vrow[j] - kv[j]) * ddelta[j];
        }
        // kv = S_d^T k_hat
        for (int i = 0; i < d.Dk; ++i)
          for (int j = 0; j < d.Dv; ++j) {
            dSh[(int64_t)i * d.Dv + j] += khat[i] * dkv[j];
            dkh[i] += Sd[(int64_t)i * d.Dv + j] * dkv[j];
          }
        // S_d = diag(g) S_prev
        for (int i = 0; i < d.Dk; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d.Dv; ++j) {
            acc += S_prev[(int64_t)i * d.Dv + j] * dSh[(int64_t)i * d.Dv + j];
            dSh[(int64_t)i * d.Dv + j] *= g[i];
          }
          dg[i] = acc;
        }
        // g = exp(l), l = -exp(a_log) softplus(x)
        for (int c = 0; c < d.Dk; ++c) {
          const double dl = dg[c] * g[c];
          const double dx = dl * (-std::exp(in.a_log[h])) * sigmoid(x[c]);
          dalpha[t * dalpha_ld + (int64_t)h * d.Dk + c] = dx;
          pb[((size_t)n * d.Hv + h) * d.Dk + c] += dx;
          pa[(size_t)n * d.Hv + h] += dl * l[c];
        }
        dbeta_raw[t * dbeta_ld + h] = db * b * (1.0 - b);
        double dot_q = 0.0, dot_k = 0.0;
        for (int i = 0; i < d.Dk; ++i) {
          dot_q += dqh[i] * qh[i];
          dot_k += dkh[i] * khat[i];
        }
        for (int i = 0; i < d.Dk; ++i) {
          dq_acc[i] += (dqh[i] - qh[i] * dot_q) / nq;
          dk_acc[i] += (dkh[i] - khat[i] * dot_k) / nk;
        }
      }
      for (int i = 0; i < d.Dk; ++i) {
        dq[t * dq_ld + (int64_t)kh * d.Dk + i] = dq_acc[i];
        dk[t * dk_ld + (int64_t)kh * d.Dk + i] = dk_acc[i];
      }
    }
    if (dS0)
      for (int hh = 0; hh < d.r; ++hh)
        std::memcpy(dS0 + ((int64_t)n * d.Hv + d.vh(kh, hh)) * SZ, &dS[hh * SZ],
                    sizeof(double) * SZ);
  });
  for (int h = 0; h < d.Hv; ++h) {
    double a = 0.0;
    for (int n = 0; n < N; ++n) a += pa[(size_t)n * d.Hv + h];
    da_log[h] = a;
    for (int c = 0; c < d.Dk; ++c) {
      double s = 0.0;
      for (int n = 0; n < N; ++n) s += pb[((size_t)n * d.Hv + h) * d.Dk + c];
      db_alpha[(int64_t)h * d.Dk + c] = s;
    }
  }
  return 0;
}
