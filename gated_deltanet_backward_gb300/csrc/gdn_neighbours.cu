// gdn_neighbours.cu -- the layer steps on either side of the recurrence: the causal
// depthwise conv1d + SiLU that turns the packed q|k|v projection into the recurrence's
// inputs, and the gated RMSNorm that turns its output o into the layer output, each
// forward and backward (lattice-inference 0.6.0, src/attention/gdn_backward.rs: the
// forward's "Causal conv1d + SiLU" and "Gated RMSNorm + output projection" steps, the
// backward's sections 5 and 2).
//
// Both stream their operands once: HBM-bound work on CUDA cores, with enough arithmetic
// per byte (a sigmoid per element, up to a dozen FMAs) that the instruction count
// matters too.  So the sigmoid is ex2.approx + rcp.approx, index arithmetic is 32-bit,
// and rows whose windows lie inside one sequence take a branch-free path.  The conv
// stages token tiles of channel slabs in shared memory through 16-byte cp.async copies
// in a multistage ring (a persistent block walks a contiguous run of tiles, two or three
// in flight while it computes one) and works on 4 channels a thread; the norm moves
// 16-byte vectors (8 bf16 or 4 fp32 values) and keeps 2-4 rows of loads in flight per
// thread.  The weight gradients (dw of the conv, d gamma of the norm) are
// reduced in a fixed order -- per thread over its tokens, per block through shared
// memory, then over blocks by a second small kernel -- so they are bit-reproducible run
// to run.
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_device.cuh"
#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

// ---- 16-byte vectors <-> fp32 ------------------------------------------------------------
template <typename T>
constexpr int kVec = 16 / (int)sizeof(T);  // channels of a 16-byte vector

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
__device__ __forceinline__ void unpack(const uint4& u, float* f, float) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4& u, float* f, __nv_bfloat16) {
  unpack_bf2(u.x, f);
  unpack_bf2(u.y, f + 2);
  unpack_bf2(u.z, f + 4);
  unpack_bf2(u.w, f + 6);
}
template <typename T>
__device__ __forceinline__ void unpack(const uint4& u, float* f) {
  unpack(u, f, T());
}
__device__ __forceinline__ uint4 pack(const float* f, float) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint4 pack(const float* f, __nv_bfloat16) {
  return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                    pack_bf2(f[6], f[7]));
}
template <typename T>
__device__ __forceinline__ uint4 pack(const float* f) {
  return pack(f, T());
}
template <typename T>
__device__ __forceinline__ uint4 ld16(const T* p) {
  return *(const uint4*)p;
}
template <typename T>
__device__ __forceinline__ void st16(T* p, const uint4& u) {
  *(uint4*)p = u;
}

// sigmoid(x) = 1 / (1 + e^-x), with e^-x = 2^(-x log2 e) from the hardware's base-2
// exponential and the reciprocal from its reciprocal approximation (each within a couple
// of ulp).  For x -> -inf the exponential overflows to +inf and the reciprocal gives 0;
// for x -> +inf it underflows to 0 and the result is 1.
__device__ __forceinline__ float sigmoid_fast(float x) {
  constexpr float kLog2e = 1.4426950408889634f;
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-x * kLog2e));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return r;
}

// ---- sequences of a varlen batch ------------------------------------------------------------
// Sequence n holding token t: the largest n < n_seqs with cu[n] <= t (empty sequences
// are skipped).  Clamped to [0, n_seqs - 1], so a malformed cu_seqlens only changes
// which inputs count as "before the start", never where a load goes.
__device__ __forceinline__ int seq_of(const int32_t* cu, int n_seqs, int t) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// ---- causal depthwise conv1d + SiLU --------------------------------------------------------
// Window entry j of row t holds input t - (K-1) + j; entries before the row's sequence
// start (j < K-1-dist, dist = t - start) are zeroed, which drops their taps from every
// product that follows.  As the window slides within a sequence those entries stay
// before its start, and a row that starts a new sequence zeroes all K-1 again.
template <int K, int V>
__device__ __forceinline__ void mask_window(float (&win)[K][V], int dist) {
  if (dist < K - 1) {
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
      if (j < K - 1 - dist)
#pragma unroll
        for (int c = 0; c < V; ++c) win[j][c] = 0.f;
  }
}

// A thread's channel vector: 4 channels (8 bytes of bf16, 16 of fp32), read from a staged
// row in shared memory and written to global memory.
__device__ __forceinline__ void ld4(const char* p, float* f, float) {
  const float4 a = *(const float4*)p;
  f[0] = a.x;
  f[1] = a.y;
  f[2] = a.z;
  f[3] = a.w;
}
__device__ __forceinline__ void ld4(const char* p, float* f, __nv_bfloat16) {
  const uint2 u = *(const uint2*)p;
  unpack_bf2(u.x, f);
  unpack_bf2(u.y, f + 2);
}
template <typename T>
__device__ __forceinline__ void ld4(const char* p, float* f) {
  ld4(p, f, T());
}
__device__ __forceinline__ void st4(float* p, const float* f) {
  *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float* f) {
  *(uint2*)p = make_uint2(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]));
}

// y[t, c] = SiLU(sum_j w[c, j] x[t - (K-1) + j, c]), inputs before the start of t's
// sequence read as zero.  The channels are cut into slabs of 1 KB rows, the tokens into
// tiles of kConvTR; tile i is token tile i % n_tt of slab i / n_tt, and block b walks
// tiles b q .. b q + q - 1 (consecutive token tiles of a slab, so the K-1 rows before a
// tile are the L2-resident end of the previous one).  A tile's rows (with the K-1 before
// it) land in a ring of kConvNS shared-memory stages through 16-byte cp.async copies,
// issued kConvNS-1 tiles ahead.  Thread (v, g) then computes the 4 channels v of the
// tile's rows g*RPT .. g*RPT+RPT-1, sliding a K-row window down them.
constexpr int kConvTR = 32;    // tokens of a forward tile
constexpr int kConvNS = 3;     // forward pipeline stages
constexpr int kConvRB = 1024;  // bytes of a forward slab row
constexpr int kConvFThreads = 512;

struct ConvArgs {
  int T, C, K, n_seqs, n_slabs, q;  // q: tiles of a block (a contiguous run, slab-major)
  const int32_t* cu;
  const void* x;
  int64_t x_ld;
  const float* w;
  const void* dy;
  int64_t dy_ld;
  void* y;  // forward: y; backward: dx
  int64_t y_ld;
  float* dw_part;  // backward: [gridDim.x, 2, slab channels, K] partial dw, or null
};

// Stages rows r0 .. r0 + ROWS - 1 (those inside [0, T)) of a slab, row bytes RB, the
// first nbytes of each (a multiple of 16), as dst[row][RB]: thread i copies the 16-byte
// vector i % (RB/16) of rows i / (RB/16), + THREADS / (RB/16), ...
template <int ROWS, int RB, int THREADS>
__device__ __forceinline__ void stage_rows(char* dst, const char* base, int64_t ld_bytes, int r0,
                                           int T, int nbytes) {
  constexpr int NV = RB / 16, RS = THREADS / NV;
  const int v = threadIdx.x % NV, row0 = threadIdx.x / NV;
  if (v * 16 >= nbytes) return;
  int src = r0 + row0;
  const char* p = base + (int64_t)src * ld_bytes + v * 16;
  char* d = dst + row0 * RB + v * 16;
  const int64_t step = RS * ld_bytes;
#pragma unroll 4
  for (int row = row0; row < ROWS; row += RS, src += RS, p += step, d += RS * RB)
    if ((unsigned)src < (unsigned)T) tc::cp_async16(d, p);
}

template <typename T, int K>
struct ConvFwdGeom {
  static constexpr int V = 4, SW = kConvRB / (int)sizeof(T);  // slab channels
  static constexpr int NTV = SW / V, RG = kConvFThreads / NTV, RPT = kConvTR / RG;
  static constexpr int ROWS = kConvTR + K - 1;  // the tile and the K-1 rows before it
  static constexpr size_t smem = (size_t)kConvNS * ROWS * kConvRB;
};

template <typename T, int K>
__global__ void __launch_bounds__(kConvFThreads, 2) k_conv_fwd(ConvArgs a) {
  using G = ConvFwdGeom<T, K>;
  constexpr int V = G::V, SW = G::SW, NTV = G::NTV, RPT = G::RPT, ROWS = G::ROWS;
  constexpr int TVB = V * (int)sizeof(T);  // bytes of a thread's vector
  extern __shared__ uint4 cstage[];        // [kConvNS][ROWS][kConvRB bytes]
  char* stg = (char*)cstage;
  const int n_tt = (a.T + kConvTR - 1) / kConvTR, total = a.n_slabs * n_tt;
  const int i0 = blockIdx.x * a.q, i1 = min(i0 + a.q, total);
  const int v = threadIdx.x % NTV, g = threadIdx.x / NTV;
  const int64_t xld = a.x_ld * (int64_t)sizeof(T);
  auto issue = [&](int i) {
    if (i < i1) {
      const int slab = i / n_tt, tt = i % n_tt, c0 = slab * SW;
      stage_rows<ROWS, kConvRB, kConvFThreads>(
          stg + ((i - i0) % kConvNS) * ROWS * kConvRB, (const char*)((const T*)a.x + c0), xld,
          tt * kConvTR - (K - 1), a.T, min(SW, a.C - c0) * (int)sizeof(T));
    }
    tc::cp_async_commit();  // possibly empty: keeps the group count uniform
  };
#pragma unroll
  for (int s = 0; s < kConvNS - 1; ++s) issue(i0 + s);
  float wt[K][V];
  int cur_slab = -1;
  for (int i = i0; i < i1; ++i) {  // uniform
    const int slab = i / n_tt, tt = i % n_tt, c0 = slab * SW;
    const bool vok = v * V < a.C - c0;
    if (slab != cur_slab) {
      cur_slab = slab;
      if (vok) {
#pragma unroll
        for (int c = 0; c < V; ++c)
#pragma unroll
          for (int j = 0; j < K; ++j) wt[j][c] = __ldg(a.w + (int64_t)(c0 + v * V + c) * K + j);
      }
    }
    issue(i + kConvNS - 1);
    tc::cp_async_wait<kConvNS - 1>();
    __syncthreads();
    const char* st = stg + ((i - i0) % kConvNS) * ROWS * kConvRB + v * TVB;
    const int tr = tt * kConvTR + g * RPT;  // first row of this thread
    if (vok && tr < a.T) {
      int n = seq_of(a.cu, a.n_seqs, tr);
      int start = __ldg(a.cu + n), end = __ldg(a.cu + n + 1);
      float win[K][V];  // rows t-K+1 .. t (stage rows g*RPT + r .. g*RPT + r + K-1)
#pragma unroll
      for (int j = 0; j < K - 1; ++j) ld4<T>(st + (g * RPT + j) * kConvRB, win[j]);
      T* yb = (T*)a.y + c0 + v * V + (int64_t)tr * a.y_ld;
      auto row = [&](int r) {
        ld4<T>(st + (g * RPT + r + K - 1) * kConvRB, win[K - 1]);
        float out[V];
#pragma unroll
        for (int c = 0; c < V; ++c) {
          float s = wt[K - 1][c] * win[K - 1][c];
#pragma unroll
          for (int j = 0; j < K - 1; ++j) s = fmaf(wt[j][c], win[j][c], s);
          out[c] = s * sigmoid_fast(s);
        }
        st4(yb + (int64_t)r * a.y_ld, out);
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
#pragma unroll
          for (int c = 0; c < V; ++c) win[j][c] = win[j + 1][c];
      };
      if (tr - (K - 1) >= start && tr + RPT <= end && tr + RPT <= a.T) {
        // the rows and their windows lie inside one sequence: no checks per row
#pragma unroll
        for (int r = 0; r < RPT; ++r) row(r);
      } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int t = tr + r;
          if (t >= a.T) break;
          while (t >= end && n + 1 < a.n_seqs) {  // next sequence
            ++n;
            start = end;
            end = __ldg(a.cu + n + 1);
          }
          mask_window<K, V>(win, t - start);  // the rows before t's start (window[0..K-2])
          row(r);
        }
      }
    }
    __syncthreads();  // the stage is refilled by a later issue
  }
  tc::cp_async_wait<0>();
}

// Backward (section 5 of the backward): d_sum[t] = dy[t] SiLU'(pre[t]) with pre[t] the
// forward's pre-activation (recomputed from x); dx[s] = sum_m d_sum[s + m] w[K-1-m] over
// the s + m inside s's sequence; dw[c, j] = sum_t d_sum[t] x[t - (K-1) + j].
// Tiles are kConvTRB tokens of a slab of 256-byte rows; a stage holds the tile's x rows
// with K-1 before and K-1 after it, and its dy rows with K-1 after it.  Phase A forms
// d_sum of the tile's rows and the K-1 after them (those once more in the next tile) into
// an fp32 shared buffer, accumulating dw over the tile's own rows; phase B reads it back
// for dx.  Block b takes tiles [b q, (b+1) q) of the slab-major tile order, so it spans
// at most two slabs: its dw is kept per slab it touches (slot 0 the first, slot 1 the
// second) and summed over blocks by k_conv_dw_sum in block order.
constexpr int kConvTRB = 64;   // tokens of a backward tile
constexpr int kConvNSB = 4;    // backward pipeline stages
constexpr int kConvRBB = 256;  // bytes of a backward slab row

template <typename T, int K>
struct ConvBwdGeom {
  static constexpr int V = 4, SW = kConvRBB / (int)sizeof(T);  // slab channels
  static constexpr int NTV = SW / V, RG = 16, THREADS = NTV * RG, RPT = kConvTRB / RG;
  static constexpr int XR = kConvTRB + 2 * (K - 1), GR = kConvTRB + (K - 1);
  static constexpr int STAGE = (XR + GR) * kConvRBB;  // bytes of a stage
  static constexpr size_t smem = (size_t)STAGE * kConvNSB + sizeof(float) * (size_t)GR * SW;
};

template <typename T, int K>
__device__ __forceinline__ void conv_dw_flush(float (&dwa)[K][4], float* red, float* part, int v,
                                              int g) {
  using G = ConvBwdGeom<T, K>;
  constexpr int V = G::V, NTV = G::NTV, KV = K * V;
  __syncthreads();  // red aliases the d_sum buffer
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int c = 0; c < V; ++c) red[(g * NTV + v) * KV + c * K + j] = dwa[j][c];
  __syncthreads();
  for (int e = threadIdx.x; e < NTV * KV; e += G::THREADS) {  // e = (vector, c, j)
    float s = 0.f;
    for (int gg = 0; gg < G::RG; ++gg) s += red[gg * NTV * KV + e];
    part[e] = s;  // [slab channel][tap]
  }
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int c = 0; c < V; ++c) dwa[j][c] = 0.f;
}

template <typename T, int K>
__global__ void __launch_bounds__(ConvBwdGeom<T, K>::THREADS, 1) k_conv_bwd(ConvArgs a) {
  using G = ConvBwdGeom<T, K>;
  constexpr int V = G::V, NTV = G::NTV, RPT = G::RPT, XR = G::XR, GR = G::GR, SW = G::SW;
  constexpr int TVB = V * (int)sizeof(T), RB = kConvRBB;
  extern __shared__ uint4 cstage[];  // [kConvNSB][XR + GR][RB bytes], then d_sum [GR][SW]
  char* stg = (char*)cstage;
  float* dsb = (float*)(stg + (size_t)G::STAGE * kConvNSB);
  const int n_tt = (a.T + kConvTRB - 1) / kConvTRB, total = a.n_slabs * n_tt;
  const int i0 = blockIdx.x * a.q, i1 = min(i0 + a.q, total);
  const int v = threadIdx.x % NTV, g = threadIdx.x / NTV;
  const int64_t xld = a.x_ld * (int64_t)sizeof(T), gld = a.dy_ld * (int64_t)sizeof(T);
  auto issue = [&](int i) {
    if (i < i1) {
      const int slab = i / n_tt, tt = i % n_tt, c0 = slab * SW, t0 = tt * kConvTRB;
      const int nb = min(SW, a.C - c0) * (int)sizeof(T);
      char* st = stg + (size_t)((i - i0) % kConvNSB) * G::STAGE;
      stage_rows<XR, RB, G::THREADS>(st, (const char*)((const T*)a.x + c0), xld, t0 - (K - 1),
                                     a.T, nb);
      stage_rows<GR, RB, G::THREADS>(st + XR * RB, (const char*)((const T*)a.dy + c0), gld, t0,
                                     a.T, nb);
    }
    tc::cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kConvNSB - 1; ++s) issue(i0 + s);
  float dwa[K][V];
#pragma unroll
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int c = 0; c < V; ++c) dwa[j][c] = 0.f;
  float wt[K][V];
  int cur_slab = -1;
  for (int i = i0; i < i1; ++i) {  // uniform
    const int slab = i / n_tt, tt = i % n_tt, c0 = slab * SW, t0 = tt * kConvTRB;
    if (slab != cur_slab) {
      if (cur_slab >= 0 && a.dw_part)  // the block's first slab ends: slot 0
        conv_dw_flush<T, K>(dwa, dsb, a.dw_part + (size_t)blockIdx.x * 2 * SW * K, v, g);
      cur_slab = slab;
      if (v * V < a.C - c0) {
#pragma unroll
        for (int c = 0; c < V; ++c)
#pragma unroll
          for (int j = 0; j < K; ++j) wt[j][c] = __ldg(a.w + (int64_t)(c0 + v * V + c) * K + j);
      }
    }
    issue(i + kConvNSB - 1);
    tc::cp_async_wait<kConvNSB - 1>();
    __syncthreads();
    const char* xs = stg + (size_t)((i - i0) % kConvNSB) * G::STAGE + v * TVB;
    const char* gs = xs + XR * RB;
    const bool vok = v * V < a.C - c0;
    // ---- phase A: d_sum of rows u = g*RPT .. g*RPT+RPT-1 (and u = kConvTRB + g, g < K-1)
    // dist: tokens of t's sequence before t
    // CHECK false: the caller knows t < T and the whole window lies in t's sequence
    auto dsum_row = [&](int u, int dist, float (&win)[K][V], bool own, auto check) {
      constexpr bool CHECK = decltype(check)::value;
      const int t = t0 + u;
      float ds[V];
      if (!CHECK || t < a.T) {
        float gy[V];
        ld4<T>(gs + u * RB, gy);
        if (CHECK) mask_window<K, V>(win, dist);
#pragma unroll
        for (int c = 0; c < V; ++c) {
          float s = wt[K - 1][c] * win[K - 1][c];
#pragma unroll
          for (int j = 0; j < K - 1; ++j) s = fmaf(wt[j][c], win[j][c], s);
          const float sg = sigmoid_fast(s);
          ds[c] = gy[c] * fmaf(s * sg, 1.f - sg, sg);  // dy * SiLU'(s)
        }
        if (own) {
#pragma unroll
          for (int j = 0; j < K; ++j)
#pragma unroll
            for (int c = 0; c < V; ++c) dwa[j][c] = fmaf(ds[c], win[j][c], dwa[j][c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < V; ++c) ds[c] = 0.f;
      }
      *(float4*)(dsb + u * SW + v * V) = make_float4(ds[0], ds[1], ds[2], ds[3]);
    };
    if (vok) {
      float win[K][V];
      const int tr = min(t0 + g * RPT, a.T - 1);
      int n = seq_of(a.cu, a.n_seqs, tr);
      int start = __ldg(a.cu + n), end = __ldg(a.cu + n + 1);
#pragma unroll
      for (int j = 0; j < K - 1; ++j) ld4<T>(xs + (g * RPT + j) * RB, win[j]);
      const int ta = t0 + g * RPT;
      if (ta - (K - 1) >= start && ta + RPT <= end && ta + RPT <= a.T) {
        // the rows and their windows lie inside one sequence: no checks per row
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int u = g * RPT + r;
          ld4<T>(xs + (u + K - 1) * RB, win[K - 1]);
          dsum_row(u, K - 1, win, true, std::false_type());
#pragma unroll
          for (int j = 0; j < K - 1; ++j)
#pragma unroll
            for (int c = 0; c < V; ++c) win[j][c] = win[j + 1][c];
        }
      } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int u = g * RPT + r, t = t0 + u;
          while (t >= end && n + 1 < a.n_seqs) {
            ++n;
            start = end;
            end = __ldg(a.cu + n + 1);
          }
          ld4<T>(xs + (u + K - 1) * RB, win[K - 1]);
          dsum_row(u, t - start, win, true, std::true_type());
#pragma unroll
          for (int j = 0; j < K - 1; ++j)
#pragma unroll
            for (int c = 0; c < V; ++c) win[j][c] = win[j + 1][c];
        }
      }
      if (g < K - 1) {  // one of the K-1 rows after the tile
        const int u = kConvTRB + g, t = min(t0 + u, a.T - 1);
#pragma unroll
        for (int j = 0; j < K; ++j) ld4<T>(xs + (u + j) * RB, win[j]);
        dsum_row(u, t - __ldg(a.cu + seq_of(a.cu, a.n_seqs, t)), win, false, std::true_type());
      }
    }
    __syncthreads();
    // ---- phase B: dx of rows s = t0 + g*RPT + r
    if (vok) {
      const int s0 = t0 + g * RPT;
      int n = seq_of(a.cu, a.n_seqs, s0 < a.T ? s0 : a.T - 1);
      int end = __ldg(a.cu + n + 1);
      T* dxb = (T*)a.y + c0 + v * V;
      // dx of row s0 + r from d_sum rows r .. r+K-1 (room: how many of them count)
      auto dx_row = [&](int r, int room) {
        float out[V];
#pragma unroll
        for (int c = 0; c < V; ++c) out[c] = 0.f;
#pragma unroll
        for (int m = 0; m < K; ++m) {
          if (m < room) {
            const float4 f = *(const float4*)(dsb + (g * RPT + r + m) * SW + v * V);
            out[0] = fmaf(f.x, wt[K - 1 - m][0], out[0]);
            out[1] = fmaf(f.y, wt[K - 1 - m][1], out[1]);
            out[2] = fmaf(f.z, wt[K - 1 - m][2], out[2]);
            out[3] = fmaf(f.w, wt[K - 1 - m][3], out[3]);
          }
        }
        st4(dxb + (int64_t)(s0 + r) * a.y_ld, out);
      };
      if (s0 + RPT - 1 + (K - 1) < end && s0 + RPT <= a.T) {
        // every row's K taps lie inside its sequence
#pragma unroll
        for (int r = 0; r < RPT; ++r) dx_row(r, K);
      } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int s = s0 + r;
          if (s >= a.T) break;
          while (s >= end && n + 1 < a.n_seqs) end = __ldg(a.cu + (++n) + 1);
          dx_row(r, end - s);
        }
      }
    }
    __syncthreads();  // d_sum buffer and stage reused
  }
  tc::cp_async_wait<0>();
  if (a.dw_part && cur_slab >= 0) {  // uniform
    const bool second = cur_slab != (i0 / n_tt);
    conv_dw_flush<T, K>(dwa, dsb, a.dw_part + ((size_t)blockIdx.x * 2 + (second ? 1 : 0)) * SW * K,
                        v, g);
  }
}

// dw[c, j] = sum over the blocks b whose tiles touch c's slab, in order, of their partial
// for that slab (slot 0 when the slab is the block's first, else slot 1).
__global__ void __launch_bounds__(256) k_conv_dw_sum(const float* part, int C, int K, int SW,
                                                     int n_tt, int q, float* dw) {
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= C * K) return;
  const int c = e / K, j = e % K, s = c / SW, cc = c % SW;
  const int b0 = (s * n_tt) / q, b1 = ((s + 1) * n_tt - 1) / q;
  float acc = 0.f;
  for (int b = b0; b <= b1; ++b) {
    const int slot = (b * q) / n_tt == s ? 0 : 1;
    acc += part[(((size_t)b * 2 + slot) * SW + cc) * K + j];
  }
  dw[e] = acc;
}

// ---- gated RMSNorm --------------------------------------------------------------------------
// Per (token t, head h) row of D values: rms = sqrt(mean o^2 + eps),
// y = (o / rms) gamma SiLU(z), gamma [D] shared by the heads.  A token's H*D values are
// H*LPR 16-byte vectors (LPR = D / V a row), numbered j; vector g of the launch is vector
// g % (H LPR) of token g / (H LPR), its column j V.  The LPR vectors of a row are
// consecutive lanes of one warp, so the row sums are butterflies over LPR lanes; a thread
// always holds the same column of gamma (vector index mod LPR = lane mod LPR).
constexpr int kNormThreads = 256;
constexpr int kNormFwdNI = 4;          // vectors of a forward thread (loads in flight)
constexpr int kNormBwdNI = 2;          // vectors of a backward thread per step
constexpr int kNormBwdMaxBlocks = 1024;

struct NormArgs {
  int T, H, D;
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

template <typename T, int LPR>
__global__ void __launch_bounds__(kNormThreads) k_norm_fwd(NormArgs a) {
  constexpr int V = kVec<T>, NI = kNormFwdNI;
  const uint32_t HV = (uint32_t)a.H * LPR, nv = (uint32_t)a.T * HV;
  const int li = threadIdx.x % LPR;
  uint4 ov[NI], zv[NI];
  uint32_t tk[NI], jv[NI];
#pragma unroll
  for (int k = 0; k < NI; ++k) {
    const uint32_t g = ((uint32_t)blockIdx.x * NI + k) * kNormThreads + threadIdx.x;
    tk[k] = g / HV;
    jv[k] = g - tk[k] * HV;
    if (g < nv) {
      ov[k] = ld16((const T*)a.o + tk[k] * a.o_ld + jv[k] * V);
      zv[k] = ld16((const T*)a.z + tk[k] * a.z_ld + jv[k] * V);
    } else {
      ov[k] = zv[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float gm[V];
#pragma unroll
  for (int c = 0; c < V; ++c) gm[c] = __ldg(a.gamma + li * V + c);
  const float invD = 1.f / (float)a.D;
#pragma unroll
  for (int k = 0; k < NI; ++k) {
    float o[V], z[V];
    unpack<T>(ov[k], o);
    unpack<T>(zv[k], z);
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) ss = fmaf(o[c], o[c], ss);
    ss = row_sum<LPR>(ss);  // every lane: the shuffles need the whole warp
    const float inv = rsqrtf(fmaf(ss, invD, a.eps));
    float y[V];
#pragma unroll
    for (int c = 0; c < V; ++c) y[c] = o[c] * inv * gm[c] * (z[c] * sigmoid_fast(z[c]));
    if (tk[k] < (uint32_t)a.T) st16((T*)a.y + tk[k] * a.y_ld + jv[k] * V, pack<T>(y));
  }
}

// Backward (section 2 of the backward): d_xn = dy gamma SiLU(z),
// dz = dy gamma x_n SiLU'(z), do = d_xn / rms - o (sum_j d_xn_j o_j) / (rms^3 D),
// d gamma = sum over rows of dy x_n SiLU(z).  Blocks take groups of NI * 256 vectors
// grid-stride (a fixed grid), so each thread's d gamma share, and the block sum over its
// row slots, have a fixed order.
template <typename T, int LPR>
__global__ void __launch_bounds__(kNormThreads, 4) k_norm_bwd(NormArgs a) {
  constexpr int V = kVec<T>, NI = kNormBwdNI, RPB = kNormThreads / LPR;
  __shared__ float red[RPB][LPR * V];
  const uint32_t HV = (uint32_t)a.H * LPR, nv = (uint32_t)a.T * HV;
  const int li = threadIdx.x % LPR, slot = threadIdx.x / LPR;
  float gm[V], dga[V];
#pragma unroll
  for (int c = 0; c < V; ++c) {
    gm[c] = __ldg(a.gamma + li * V + c);
    dga[c] = 0.f;
  }
  const float invD = 1.f / (float)a.D;
  const uint32_t n_groups = (nv + NI * kNormThreads - 1) / (NI * kNormThreads);
  for (uint32_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {  // uniform per block
    uint4 ov[NI], zv[NI], gv[NI];
    uint32_t tk[NI], jv[NI];
#pragma unroll
    for (int k = 0; k < NI; ++k) {
      const uint32_t g = (grp * NI + k) * kNormThreads + threadIdx.x;
      tk[k] = g / HV;
      jv[k] = g - tk[k] * HV;
      if (g < nv) {
        ov[k] = ld16((const T*)a.o + tk[k] * a.o_ld + jv[k] * V);
        zv[k] = ld16((const T*)a.z + tk[k] * a.z_ld + jv[k] * V);
        gv[k] = ld16((const T*)a.dy + tk[k] * a.dy_ld + jv[k] * V);
      } else {
        ov[k] = zv[k] = gv[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int k = 0; k < NI; ++k) {
      float o[V], z[V], dy[V];
      unpack<T>(ov[k], o);
      unpack<T>(zv[k], z);
      unpack<T>(gv[k], dy);
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < V; ++c) ss = fmaf(o[c], o[c], ss);
      ss = row_sum<LPR>(ss);
      const float inv = rsqrtf(fmaf(ss, invD, a.eps));
      float dxn[V], dz[V], dot = 0.f;
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const float sg = sigmoid_fast(z[c]), sz = z[c] * sg;
        const float xn = o[c] * inv, dyg = dy[c] * gm[c];
        dxn[c] = dyg * sz;
        dz[c] = dyg * xn * fmaf(sz, 1.f - sg, sg);  // SiLU'(z) = sg + z sg (1 - sg)
        dga[c] = fmaf(dy[c] * xn, sz, dga[c]);
        dot = fmaf(dxn[c], o[c], dot);
      }
      dot = row_sum<LPR>(dot);
      const float cc = dot * inv * inv * inv * invD;
      if (tk[k] < (uint32_t)a.T) {
        float d_o[V];
#pragma unroll
        for (int c = 0; c < V; ++c) d_o[c] = fmaf(dxn[c], inv, -o[c] * cc);
        st16((T*)a.y + tk[k] * a.y_ld + jv[k] * V, pack<T>(d_o));
        st16((T*)a.dz + tk[k] * a.dz_ld + jv[k] * V, pack<T>(dz));
      }
    }
  }
  if (!a.dg_part) return;  // uniform
#pragma unroll
  for (int c = 0; c < V; ++c) red[slot][li * V + c] = dga[c];
  __syncthreads();
  for (int j = threadIdx.x; j < a.D; j += kNormThreads) {
    float s = 0.f;
    for (int sl = 0; sl < RPB; ++sl) s += red[sl][j];
    a.dg_part[(size_t)blockIdx.x * a.D + j] = s;
  }
}

// d gamma[i] = sum over blocks b in order of part[b, i]: one warp per output, lane l
// summing b = l, l + 32, ... in order, then a butterfly over the lanes (a fixed order).
__global__ void __launch_bounds__(256) k_sum_parts_warp(const float* part, int nb, int n,
                                                        float* out) {
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;  // whole warps
  float s = 0.f;
  for (int b = lane; b < nb; b += 32) s += part[(size_t)b * n + i];
  out[i] = warp_sum(s);
}

// ---- launch geometry ------------------------------------------------------------------------
struct ConvGeom {
  int n_slabs, n_tt, total, q, grid;
};
// Forward: 2 blocks an SM; backward: 1 block an SM and at most 2 slabs a block (q <= n_tt).
// `blocks` is the number of resident blocks to fill (capped at 1024).
inline ConvGeom conv_geom(bool bwd, int T, int C, int es, int blocks) {
  ConvGeom g;
  const int sw = (bwd ? kConvRBB : kConvRB) / es;  // slab channels
  const int tr = bwd ? kConvTRB : kConvTR;
  g.n_slabs = (C + sw - 1) / sw;
  g.n_tt = (T + tr - 1) / tr;
  g.total = g.n_slabs * g.n_tt;
  blocks = blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks);
  g.q = (g.total + blocks - 1) / blocks;
  if (bwd && g.q > g.n_tt) g.q = g.n_tt;
  if (g.q < 1) g.q = 1;
  g.grid = (g.total + g.q - 1) / g.q;
  return g;
}

template <bool BWD, typename T, int K>
cudaError_t conv_launch(const ConvArgs& a, int grid, cudaStream_t st) {
  const size_t smem = BWD ? ConvBwdGeom<T, K>::smem : ConvFwdGeom<T, K>::smem;
  const int threads = BWD ? ConvBwdGeom<T, K>::THREADS : kConvFThreads;
  static bool attr_set = false;  // one instantiation, one attribute
  if (!attr_set) {
    const cudaError_t e =
        BWD ? cudaFuncSetAttribute(k_conv_bwd<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem)
            : cudaFuncSetAttribute(k_conv_fwd<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if constexpr (BWD)
    k_conv_bwd<T, K><<<grid, threads, smem, st>>>(a);
  else
    k_conv_fwd<T, K><<<grid, threads, smem, st>>>(a);
  return cudaGetLastError();
}

template <bool BWD, typename T>
cudaError_t conv_dispatch(int K, const ConvArgs& a, int grid, cudaStream_t st) {
  switch (K) {
    case 1: return conv_launch<BWD, T, 1>(a, grid, st);
    case 2: return conv_launch<BWD, T, 2>(a, grid, st);
    case 3: return conv_launch<BWD, T, 3>(a, grid, st);
    case 4: return conv_launch<BWD, T, 4>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BWD, typename T>
cudaError_t norm_dispatch(const NormArgs& a, int grid, cudaStream_t st) {
  const int LPR = a.D / kVec<T>;
#define GDN_NORM_CASE(L)                                      \
  case L:                                                     \
    if constexpr (BWD)                                        \
      k_norm_bwd<T, L><<<grid, kNormThreads, 0, st>>>(a);     \
    else                                                      \
      k_norm_fwd<T, L><<<grid, kNormThreads, 0, st>>>(a);     \
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

template <typename T>
int norm_bwd_resident_blocks(int D) {
  int per_sm = 0;
  const int LPR = D / kVec<T>;
  cudaError_t e = cudaErrorInvalidValue;
  switch (LPR) {
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_norm_bwd<T, 2>, kNormThreads, 0); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_norm_bwd<T, 4>, kNormThreads, 0); break;
    case 8: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_norm_bwd<T, 8>, kNormThreads, 0); break;
    case 16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_norm_bwd<T, 16>, kNormThreads, 0); break;
    case 32: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_norm_bwd<T, 32>, kNormThreads, 0); break;
    default: break;
  }
  if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  return per_sm * sm_count();
}

}  // namespace

size_t conv_partial_floats(int64_t T, int C, int K) {
  // the largest backward grid any device could get (1024 resident blocks), either dtype
  size_t most = 0;
  for (int es : {2, 4}) {
    const ConvGeom g = conv_geom(true, (int)T, C, es, 1024);
    const size_t f = (size_t)g.grid * 2 * (kConvRBB / es) * K;
    most = f > most ? f : most;
  }
  return most;
}
size_t norm_partial_floats(int D) { return (size_t)kNormBwdMaxBlocks * (size_t)D; }

cudaError_t launch_conv1d_silu(bool bwd, int dtype, int64_t T, int C, int K, const int32_t* cu,
                               int n_seqs, const void* x, int64_t x_ld, const float* w,
                               const void* dy, int64_t dy_ld, void* y, int64_t y_ld, float* dw,
                               float* part, cudaStream_t st) {
  const bool bf = dtype == GDN_DTYPE_BF16;
  const int es = bf ? 2 : 4;
  const ConvGeom g = conv_geom(bwd, (int)T, C, es, (bwd ? 1 : 2) * sm_count());
  ConvArgs a;
  a.T = (int)T;
  a.C = C;
  a.K = K;
  a.n_seqs = n_seqs;
  a.n_slabs = g.n_slabs;
  a.q = g.q;
  a.cu = cu;
  a.x = x;
  a.x_ld = x_ld;
  a.w = w;
  a.dy = dy;
  a.dy_ld = dy_ld;
  a.y = y;
  a.y_ld = y_ld;
  a.dw_part = bwd && dw ? part : nullptr;
  profile_pre(st, bwd ? KID_CONV_BWD : KID_CONV_FWD);
  cudaError_t e;
  if (bwd)
    e = bf ? conv_dispatch<true, __nv_bfloat16>(K, a, g.grid, st)
           : conv_dispatch<true, float>(K, a, g.grid, st);
  else
    e = bf ? conv_dispatch<false, __nv_bfloat16>(K, a, g.grid, st)
           : conv_dispatch<false, float>(K, a, g.grid, st);
  profile_post(st);
  if (e != cudaSuccess || !a.dw_part) return e;
  profile_pre(st, KID_SUM_PARTS);
  k_conv_dw_sum<<<(C * K + 255) / 256, 256, 0, st>>>(part, C, K, kConvRBB / es, g.n_tt,
                                                     g.q, dw);
  profile_post(st);
  return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(bool bwd, int dtype, int64_t T, int H, int D, float eps,
                                 const void* o, int64_t o_ld, const void* z, int64_t z_ld,
                                 const float* gamma, const void* dy, int64_t dy_ld, void* y,
                                 int64_t y_ld, void* dz, int64_t dz_ld, float* dgamma,
                                 float* part, cudaStream_t st) {
  NormArgs a;
  a.T = (int)T;
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
  const int64_t nv = T * H * (D / (bf ? 8 : 4));  // 16-byte vectors
  const int NI = bwd ? kNormBwdNI : kNormFwdNI;
  const int64_t groups = (nv + NI * kNormThreads - 1) / (NI * kNormThreads);
  int grid = (int)groups;
  if (bwd) {
    int res = bf ? norm_bwd_resident_blocks<__nv_bfloat16>(D) : norm_bwd_resident_blocks<float>(D);
    res = res > kNormBwdMaxBlocks ? kNormBwdMaxBlocks : res;
    grid = groups < res ? (int)groups : res;
  }
  profile_pre(st, bwd ? KID_NORM_BWD : KID_NORM_FWD);
  cudaError_t e;
  if (bwd)
    e = bf ? norm_dispatch<true, __nv_bfloat16>(a, grid, st) : norm_dispatch<true, float>(a, grid, st);
  else
    e = bf ? norm_dispatch<false, __nv_bfloat16>(a, grid, st)
           : norm_dispatch<false, float>(a, grid, st);
  profile_post(st);
  if (e != cudaSuccess || !a.dg_part) return e;
  profile_pre(st, KID_SUM_PARTS);
  k_sum_parts_warp<<<(D + 7) / 8, 256, 0, st>>>(part, grid, D, dgamma);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
