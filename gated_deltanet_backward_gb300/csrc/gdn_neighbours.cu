// gdn_neighbours.cu -- the layer steps on either side of the recurrence: the causal
// depthwise conv1d + SiLU that turns the packed q|k|v projection into the recurrence's
// inputs, and the gated RMSNorm that turns its output o into the layer output, each
// forward and backward (lattice-inference 0.6.0, src/attention/gdn_backward.rs: the
// forward's "Causal conv1d + SiLU" and "Gated RMSNorm + output projection" steps, the
// backward's sections 5 and 2).
//
// Both are elementwise or row-local and stream their operands once: HBM-bound work on
// CUDA cores.  Every thread moves vectors of 4 or 8 channels (8 or 16 bytes), so a warp
// covers 256 or 512 contiguous bytes of a row, and the weight gradients (dw of the conv,
// d gamma of the norm) are reduced in a fixed order -- per thread over its tokens, per
// block over its warps or row slots through shared memory, then over blocks by a
// second small kernel -- so they are bit-reproducible run to run.
#include <cuda_bf16.h>

#include "gdn_device.cuh"
#include "gdn_internal.cuh"

namespace gdn {
namespace {

// ---- vectors of V channels (8 or 16 bytes), converted to and from fp32 ------------------
template <typename T, int V>
struct Vec;
template <>
struct Vec<float, 4> {
  __device__ __forceinline__ static void load(const float* p, float* f) {
    const float4 a = *(const float4*)p;
    f[0] = a.x;
    f[1] = a.y;
    f[2] = a.z;
    f[3] = a.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* f) {
    *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
  }
};
__device__ __forceinline__ void unpack_bf2(uint32_t w, float* f) {
  __nv_bfloat162 b;
  memcpy(&b, &w, 4);
  const float2 x = __bfloat1622float2(b);
  f[0] = x.x;
  f[1] = x.y;
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  uint32_t w;
  memcpy(&w, &h, 4);
  return w;
}
template <>
struct Vec<__nv_bfloat16, 8> {
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* f) {
    const uint4 u = *(const uint4*)p;
    unpack_bf2(u.x, f);
    unpack_bf2(u.y, f + 2);
    unpack_bf2(u.z, f + 4);
    unpack_bf2(u.w, f + 6);
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* f) {
    *(uint4*)p = make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                            pack_bf2(f[6], f[7]));
  }
};
template <>
struct Vec<__nv_bfloat16, 4> {
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* f) {
    const uint2 u = *(const uint2*)p;
    unpack_bf2(u.x, f);
    unpack_bf2(u.y, f + 2);
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* f) {
    *(uint2*)p = make_uint2(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]));
  }
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + expf(-x)); }
// d/dx x sigmoid(x) = sigmoid(x) (1 + x (1 - sigmoid(x)))
__device__ __forceinline__ float silu_grad_f(float x) {
  const float s = 1.f / (1.f + expf(-x));
  return s * (1.f + x * (1.f - s));
}

// ---- causal depthwise conv1d + SiLU --------------------------------------------------------
// y[t, c] = SiLU(sum_j w[c, j] x[t - (K-1) + j, c]), inputs before the start of t's
// sequence read as zero.  A block is 8 warps: lane l takes the channel vector (V channels)
// 32 * blockIdx.x + l, warp i the kConvTT tokens starting at 256 * blockIdx.y + kConvTT i.
// A thread walks its tokens in order, holding the K-1 previous inputs in registers and
// issuing the loads of U tokens ahead.
constexpr int kConvWarps = 8;
constexpr int kConvTT = 32;                     // tokens of one warp
constexpr int kConvRows = kConvWarps * kConvTT; // tokens of one block

struct ConvArgs {
  int64_t T;
  int C, n_seqs;
  const int32_t* cu;
  const void* x;
  int64_t x_ld;
  const float* w;
  const void* dy;
  int64_t dy_ld;
  void* y;  // forward: y; backward: dx
  int64_t y_ld;
  float* dw_part;  // backward: [ceil(T / kConvRows), C, K] partial dw, or null
};

// Sequence n holding token t: the largest n < n_seqs with cu[n] <= t (empty sequences
// are skipped).  Clamped to [0, n_seqs - 1], so a malformed cu_seqlens only changes
// which inputs count as "before the start", never where a load goes.
__device__ __forceinline__ int seq_of(const int32_t* cu, int n_seqs, int64_t t) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Steps the sequence cursor (n, end = cu[n + 1]) forward until it holds token t; true
// when it moved (t is then the first token of its sequence).
__device__ __forceinline__ bool seq_advance(const int32_t* cu, int n_seqs, int64_t t, int& n,
                                            int64_t& end) {
  bool moved = false;
  while (t >= end && n + 1 < n_seqs) {
    ++n;
    end = __ldg(cu + n + 1);
    moved = true;
  }
  return moved;
}

template <typename T, int V, int K, int U>
__global__ void __launch_bounds__(kConvWarps * 32, 2) k_conv_fwd(ConvArgs a) {
  using VT = Vec<T, V>;
  constexpr int KR = K > 1 ? K - 1 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = (blockIdx.x * 32 + lane) * V;
  const int64_t t0 = (int64_t)blockIdx.y * kConvRows + warp * kConvTT;
  if (c0 >= a.C || t0 >= a.T) return;
  const int64_t t1 = t0 + kConvTT < a.T ? t0 + kConvTT : a.T;
  const T* x = (const T*)a.x + c0;
  T* y = (T*)a.y + c0;
  float wt[K][V];
#pragma unroll
  for (int i = 0; i < V; ++i)
#pragma unroll
    for (int j = 0; j < K; ++j) wt[j][i] = __ldg(a.w + (int64_t)(c0 + i) * K + j);
  int n = seq_of(a.cu, a.n_seqs, t0);
  int64_t start = __ldg(a.cu + n), end = __ldg(a.cu + n + 1);
  float ring[KR][V];  // inputs t-K+1 .. t-1 (zero before the sequence start)
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int64_t src = t0 - (K - 1) + j;
    if (src >= start && src >= 0)
      VT::load(x + src * a.x_ld, ring[j]);
    else
#pragma unroll
      for (int i = 0; i < V; ++i) ring[j][i] = 0.f;
  }
  for (int64_t tb = t0; tb < t1; tb += U) {
    float xv[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (tb + u < t1) VT::load(x + (tb + u) * a.x_ld, xv[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = tb + u;
      if (t >= t1) break;
      if (seq_advance(a.cu, a.n_seqs, t, n, end)) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
#pragma unroll
          for (int i = 0; i < V; ++i) ring[j][i] = 0.f;
      }
      float out[V];
#pragma unroll
      for (int i = 0; i < V; ++i) {
        float s = wt[K - 1][i] * xv[u][i];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) s = fmaf(wt[j][i], ring[j][i], s);
        out[i] = silu_f(s);
      }
      VT::store(y + t * a.y_ld, out);
#pragma unroll
      for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
        for (int i = 0; i < V; ++i) ring[j][i] = ring[j + 1][i];
      if (K > 1)
#pragma unroll
        for (int i = 0; i < V; ++i) ring[KR - 1][i] = xv[u][i];
    }
  }
}

// Backward (section 5 of the backward): d_sum[t] = dy[t] SiLU'(pre[t]) with pre[t] the
// forward's pre-activation (recomputed); dx[s] = sum_m d_sum[s + m] w[K-1-m] over the
// s + m inside s's sequence; dw[c, j] = sum_t d_sum[t] x[t - (K-1) + j].  A warp's
// tokens s are [t0, t1); it walks t from t0 to t1 + K - 2 (the K-1 tokens after t1 are
// recomputed, not counted into dw), holding the K-1 previous inputs and d_sums.
template <typename T, int V, int K, int U>
__global__ void __launch_bounds__(kConvWarps * 32, 2) k_conv_bwd(ConvArgs a) {
  using VT = Vec<T, V>;
  constexpr int KR = K > 1 ? K - 1 : 1;
  __shared__ float red[kConvWarps][K * V][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = (blockIdx.x * 32 + lane) * V;
  const int64_t t0 = (int64_t)blockIdx.y * kConvRows + warp * kConvTT;
  float dwa[K][V];
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int i = 0; i < V; ++i) dwa[j][i] = 0.f;
  if (c0 < a.C && t0 < a.T) {
    const int64_t t1 = t0 + kConvTT < a.T ? t0 + kConvTT : a.T;
    const int64_t te = t1 + (K - 1);  // walk end (exclusive)
    const T* x = (const T*)a.x + c0;
    const T* dy = (const T*)a.dy + c0;
    T* dx = (T*)a.y + c0;
    float wt[K][V];
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
      for (int j = 0; j < K; ++j) wt[j][i] = __ldg(a.w + (int64_t)(c0 + i) * K + j);
    int nt = seq_of(a.cu, a.n_seqs, t0);
    int64_t end_t = __ldg(a.cu + nt + 1);
    const int64_t start0 = __ldg(a.cu + nt);
    int ns = nt;  // sequence of the token s whose dx is emitted next
    int64_t end_s = end_t;
    float xr[KR][V], dr[KR][V];  // inputs t-K+1 .. t-1; d_sum of t-K+1 .. t-1
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      const int64_t src = t0 - (K - 1) + j;
      if (src >= start0 && src >= 0)
        VT::load(x + src * a.x_ld, xr[j]);
      else
#pragma unroll
        for (int i = 0; i < V; ++i) xr[j][i] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) dr[j][i] = 0.f;
    }
    for (int64_t tb = t0; tb < te; tb += U) {
      float xv[U][V], gv[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (tb + u < te && tb + u < a.T) {
          VT::load(x + (tb + u) * a.x_ld, xv[u]);
          VT::load(dy + (tb + u) * a.dy_ld, gv[u]);
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t t = tb + u;
        if (t >= te) break;
        float ds[V];
        if (t < a.T) {
          if (seq_advance(a.cu, a.n_seqs, t, nt, end_t)) {
#pragma unroll
            for (int j = 0; j < K - 1; ++j)
#pragma unroll
              for (int i = 0; i < V; ++i) xr[j][i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < V; ++i) {
            float s = wt[K - 1][i] * xv[u][i];
#pragma unroll
            for (int j = 0; j < K - 1; ++j) s = fmaf(wt[j][i], xr[j][i], s);
            ds[i] = gv[u][i] * silu_grad_f(s);
          }
          if (t < t1) {
#pragma unroll
            for (int i = 0; i < V; ++i) {
#pragma unroll
              for (int j = 0; j < K - 1; ++j) dwa[j][i] = fmaf(ds[i], xr[j][i], dwa[j][i]);
              dwa[K - 1][i] = fmaf(ds[i], xv[u][i], dwa[K - 1][i]);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) ds[i] = 0.f;
        }
        const int64_t s = t - (K - 1);
        if (s >= t0) {
          seq_advance(a.cu, a.n_seqs, s, ns, end_s);
          float out[V];
#pragma unroll
          for (int i = 0; i < V; ++i) out[i] = s + (K - 1) < end_s ? ds[i] * wt[0][i] : 0.f;
#pragma unroll
          for (int m = 0; m < K - 1; ++m)
            if (s + m < end_s)
#pragma unroll
              for (int i = 0; i < V; ++i) out[i] = fmaf(dr[m][i], wt[K - 1 - m][i], out[i]);
          VT::store(dx + s * a.y_ld, out);
        }
#pragma unroll
        for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
          for (int i = 0; i < V; ++i) {
            xr[j][i] = xr[j + 1][i];
            dr[j][i] = dr[j + 1][i];
          }
        if (K > 1)
#pragma unroll
          for (int i = 0; i < V; ++i) {
            xr[KR - 1][i] = t < a.T ? xv[u][i] : 0.f;
            dr[KR - 1][i] = ds[i];
          }
      }
    }
  }
  if (!a.dw_part) return;  // uniform: the same for every thread of the launch
  // dw of the block's tokens: warps summed in order through shared memory
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int i = 0; i < V; ++i) red[warp][i * K + j][lane] = dwa[j][i];
  __syncthreads();
  float* part = a.dw_part + (int64_t)blockIdx.y * a.C * K;
  const int64_t cb = (int64_t)blockIdx.x * 32 * V;  // first channel of the block
  for (int e = threadIdx.x; e < 32 * K * V; e += kConvWarps * 32) {
    const int l = e / (K * V), ij = e % (K * V);   // lane l, channel c0(l) + i, tap j
    const int64_t c = cb + (int64_t)l * V + ij / K;
    if (c >= a.C) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConvWarps; ++w) s += red[w][ij][l];
    part[c * K + ij % K] = s;
  }
}

// ---- gated RMSNorm --------------------------------------------------------------------------
// Per (token t, head h) row of D values: rms = sqrt(mean o^2 + eps),
// y = (o / rms) gamma SiLU(z), gamma [D] shared by the heads.  LPR = D / V lanes own a
// row (V channels each, 16 bytes); a warp holds 32 / LPR rows; the row sums are
// butterfly shuffles inside the LPR lanes.
constexpr int kNormThreads = 256;
constexpr int kNormBwdBlocks = 608;  // grid cap of the backward (fixed: d gamma's order)

struct NormArgs {
  int64_t rows;  // T * H
  int H, D;
  float eps;
  const void* o;
  int64_t o_ld;
  const void* z;
  int64_t z_ld;
  const float* gamma;
  const void* dy;
  int64_t dy_ld;
  void* y;  // forward: y; backward: do
  int64_t y_ld;
  void* dz;
  int64_t dz_ld;
  float* dg_part;  // backward: [gridDim.x, D] partial d gamma, or null
};

template <int LPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

template <typename T, int V, int LPR>
__global__ void __launch_bounds__(kNormThreads) k_norm_fwd(NormArgs a) {
  using VT = Vec<T, V>;
  const int64_t g = (int64_t)blockIdx.x * kNormThreads + threadIdx.x;
  const int64_t r = g / LPR;
  const int li = (int)(g % LPR);
  const bool ok = r < a.rows;  // every lane joins the shuffles
  const int64_t t = ok ? r / a.H : 0;
  const int h = ok ? (int)(r % a.H) : 0;
  const int64_t col = (int64_t)h * a.D + li * V;
  float o[V], z[V];
  if (ok) {
    VT::load((const T*)a.o + t * a.o_ld + col, o);
    VT::load((const T*)a.z + t * a.z_ld + col, z);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = z[i] = 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) ss = fmaf(o[i], o[i], ss);
  ss = row_sum<LPR>(ss);
  const float inv = 1.f / sqrtf(ss / (float)a.D + a.eps);
  if (!ok) return;
  float y[V];
#pragma unroll
  for (int i = 0; i < V; ++i) y[i] = o[i] * inv * __ldg(a.gamma + li * V + i) * silu_f(z[i]);
  VT::store((T*)a.y + t * a.y_ld + col, y);
}

// Backward (section 2 of the backward): d_xn = dy gamma SiLU(z),
// dz = dy gamma x_n SiLU'(z), do = d_xn / rms - o (sum_j d_xn_j o_j) / (rms^3 D),
// d gamma = sum over rows of dy x_n SiLU(z).  Rows are taken grid-stride (a fixed grid),
// so each thread's d gamma share, and the block sum over its row slots, have a fixed order.
template <typename T, int V, int LPR>
__global__ void __launch_bounds__(kNormThreads) k_norm_bwd(NormArgs a) {
  using VT = Vec<T, V>;
  constexpr int RPB = kNormThreads / LPR;  // row slots of a block
  __shared__ float red[RPB][LPR * V];
  const int li = threadIdx.x % LPR, slot = threadIdx.x / LPR;
  float dga[V];
#pragma unroll
  for (int i = 0; i < V; ++i) dga[i] = 0.f;
  float gm[V];
#pragma unroll
  for (int i = 0; i < V; ++i) gm[i] = __ldg(a.gamma + li * V + i);
  const int64_t n_groups = (a.rows + RPB - 1) / RPB;
  for (int64_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {  // uniform per block
    const int64_t r = grp * RPB + slot;
    const bool ok = r < a.rows;
    const int64_t t = ok ? r / a.H : 0;
    const int h = ok ? (int)(r % a.H) : 0;
    const int64_t col = (int64_t)h * a.D + li * V;
    float o[V], z[V], dy[V];
    if (ok) {
      VT::load((const T*)a.o + t * a.o_ld + col, o);
      VT::load((const T*)a.z + t * a.z_ld + col, z);
      VT::load((const T*)a.dy + t * a.dy_ld + col, dy);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = z[i] = dy[i] = 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) ss = fmaf(o[i], o[i], ss);
    ss = row_sum<LPR>(ss);
    const float rms = sqrtf(ss / (float)a.D + a.eps), inv = 1.f / rms;
    float dxn[V], dz[V], dot = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const float xn = o[i] * inv, sz = silu_f(z[i]);
      dxn[i] = dy[i] * gm[i] * sz;
      dz[i] = dy[i] * gm[i] * xn * silu_grad_f(z[i]);
      dga[i] = fmaf(dy[i] * xn, sz, dga[i]);
      dot = fmaf(dxn[i], o[i], dot);
    }
    dot = row_sum<LPR>(dot);
    const float c = dot * inv * inv * inv / (float)a.D;
    if (ok) {
      float d_o[V];
#pragma unroll
      for (int i = 0; i < V; ++i) d_o[i] = fmaf(dxn[i], inv, -o[i] * c);
      VT::store((T*)a.y + t * a.y_ld + col, d_o);
      VT::store((T*)a.dz + t * a.dz_ld + col, dz);
    }
  }
  if (!a.dg_part) return;  // uniform
#pragma unroll
  for (int i = 0; i < V; ++i) red[slot][li * V + i] = dga[i];
  __syncthreads();
  for (int j = threadIdx.x; j < a.D; j += kNormThreads) {
    float s = 0.f;
    for (int sl = 0; sl < RPB; ++sl) s += red[sl][j];
    a.dg_part[(int64_t)blockIdx.x * a.D + j] = s;
  }
}

// ---- fixed-order sums of per-block partials: out[i] = sum_b part[b * n + i] -------------
// Few blocks (the conv's token tiles): one thread per output, b in order.
__global__ void __launch_bounds__(256) k_sum_parts_thread(const float* part, int nb, int64_t n,
                                                          float* out) {
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int b = 0; b < nb; ++b) s += part[(int64_t)b * n + i];
  out[i] = s;
}
// Many blocks (the norm's grid): one warp per output, lane l summing b = l, l + 32, ...
// in order, then a butterfly over the lanes (a fixed order too).
__global__ void __launch_bounds__(256) k_sum_parts_warp(const float* part, int nb, int64_t n,
                                                        float* out) {
  const int64_t i = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;  // whole warps
  float s = 0.f;
  for (int b = lane; b < nb; b += 32) s += part[(int64_t)b * n + i];
  out[i] = warp_sum(s);
}

template <bool BWD, typename T, int V, int U>
cudaError_t conv_dispatch(int K, const ConvArgs& a, dim3 grid, cudaStream_t st) {
  const dim3 block(kConvWarps * 32);
#define GDN_CONV_CASE(KK)                                \
  case KK:                                               \
    if constexpr (BWD)                                   \
      k_conv_bwd<T, V, KK, U><<<grid, block, 0, st>>>(a); \
    else                                                 \
      k_conv_fwd<T, V, KK, U><<<grid, block, 0, st>>>(a); \
    break;
  switch (K) {
    GDN_CONV_CASE(1)
    GDN_CONV_CASE(2)
    GDN_CONV_CASE(3)
    GDN_CONV_CASE(4)
    default: return cudaErrorInvalidValue;
  }
#undef GDN_CONV_CASE
  return cudaGetLastError();
}

template <typename T, int V>
cudaError_t norm_dispatch(bool bwd, const NormArgs& a, cudaStream_t st) {
  const int LPR = a.D / V;
  const int64_t threads = a.rows * LPR;
  const int64_t n_groups = (a.rows + kNormThreads / LPR - 1) / (kNormThreads / LPR);
  const unsigned grid = bwd ? (unsigned)(n_groups < kNormBwdBlocks ? n_groups : kNormBwdBlocks)
                            : (unsigned)((threads + kNormThreads - 1) / kNormThreads);
#define GDN_NORM_CASE(L)                                                  \
  case L:                                                                 \
    if (bwd)                                                              \
      k_norm_bwd<T, V, L><<<grid, kNormThreads, 0, st>>>(a);              \
    else                                                                  \
      k_norm_fwd<T, V, L><<<grid, kNormThreads, 0, st>>>(a);              \
    break;
  switch (LPR) {
    GDN_NORM_CASE(2)
    GDN_NORM_CASE(4)
    GDN_NORM_CASE(8)
    GDN_NORM_CASE(16)
    GDN_NORM_CASE(32)
    default: return cudaErrorInvalidValue;
  }
#undef GDN_NORM_CASE
  return cudaGetLastError();
}

}  // namespace

size_t conv_partial_floats(int64_t T, int C, int K) {
  return (size_t)((T + kConvRows - 1) / kConvRows) * (size_t)C * (size_t)K;
}
size_t norm_partial_floats(int D) { return (size_t)kNormBwdBlocks * (size_t)D; }

cudaError_t launch_conv1d_silu(bool bwd, int dtype, int64_t T, int C, int K, const int32_t* cu,
                               int n_seqs, const void* x, int64_t x_ld, const float* w,
                               const void* dy, int64_t dy_ld, void* y, int64_t y_ld, float* dw,
                               float* part, cudaStream_t st) {
  ConvArgs a;
  a.T = T;
  a.C = C;
  a.n_seqs = n_seqs;
  a.cu = cu;
  a.x = x;
  a.x_ld = x_ld;
  a.w = w;
  a.dy = dy;
  a.dy_ld = dy_ld;
  a.y = y;
  a.y_ld = y_ld;
  a.dw_part = dw ? part : nullptr;
  // forward: 16-byte vectors, 32 bytes of loads ahead (bf16) or 64 (fp32); backward: 4
  // channels a thread and 2 tokens ahead (the walk holds twice the forward's registers)
  const bool bf = dtype == GDN_DTYPE_BF16;
  const int V = bwd ? 4 : (bf ? 8 : 4);
  const int n_tiles = (int)((T + kConvRows - 1) / kConvRows);
  const dim3 grid((unsigned)((C / V + 31) / 32), (unsigned)n_tiles);
  profile_pre(st, bwd ? KID_CONV_BWD : KID_CONV_FWD);
  cudaError_t e;
  if (bwd)
    e = bf ? conv_dispatch<true, __nv_bfloat16, 4, 2>(K, a, grid, st)
           : conv_dispatch<true, float, 4, 2>(K, a, grid, st);
  else
    e = bf ? conv_dispatch<false, __nv_bfloat16, 8, 2>(K, a, grid, st)
           : conv_dispatch<false, float, 4, 4>(K, a, grid, st);
  profile_post(st);
  if (e != cudaSuccess || !a.dw_part) return e;
  const int64_t n = (int64_t)C * K;
  profile_pre(st, KID_SUM_PARTS);
  k_sum_parts_thread<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(part, n_tiles, n, dw);
  profile_post(st);
  return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(bool bwd, int dtype, int64_t T, int H, int D, float eps,
                                 const void* o, int64_t o_ld, const void* z, int64_t z_ld,
                                 const float* gamma, const void* dy, int64_t dy_ld, void* y,
                                 int64_t y_ld, void* dz, int64_t dz_ld, float* dgamma,
                                 float* part, cudaStream_t st) {
  NormArgs a;
  a.rows = T * H;
  a.H = H;
  a.D = D;
  a.eps = eps;
  a.o = o;
  a.o_ld = o_ld;
  a.z = z;
  a.z_ld = z_ld;
  a.gamma = gamma;
  a.dy = dy;
  a.dy_ld = dy_ld;
  a.y = y;
  a.y_ld = y_ld;
  a.dz = dz;
  a.dz_ld = dz_ld;
  a.dg_part = bwd && dgamma ? part : nullptr;
  const bool bf = dtype == GDN_DTYPE_BF16;
  profile_pre(st, bwd ? KID_NORM_BWD : KID_NORM_FWD);
  const cudaError_t e = bf ? norm_dispatch<__nv_bfloat16, 8>(bwd, a, st)
                           : norm_dispatch<float, 4>(bwd, a, st);
  profile_post(st);
  if (e != cudaSuccess || !a.dg_part) return e;
  const int V = bf ? 8 : 4, LPR = D / V;
  const int64_t n_groups = (a.rows + kNormThreads / LPR - 1) / (kNormThreads / LPR);
  const int nb = (int)(n_groups < kNormBwdBlocks ? n_groups : kNormBwdBlocks);
  profile_pre(st, KID_SUM_PARTS);
  k_sum_parts_warp<<<(unsigned)((D + 7) / 8), 256, 0, st>>>(part, nb, D, dgamma);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
