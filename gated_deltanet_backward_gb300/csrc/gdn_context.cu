// gdn_context.cu -- composing segment state maps, for context parallelism: a sequence cut
// into segments maps each segment's start state affinely to its end state,
// S_out = Phi S_in + R (the forward recap's token update of lattice-inference 0.6.0,
// src/attention/gdn_backward.rs, rewritten as S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} +
// beta_t k_t v_t^T), and the start-state gradient the other way, dS_in = Phi^T dS_out + G.
// One launch applies out = op(Phi) S + R to n independent (sequence, head) blocks.
//
// A [Dk, Dk] x [Dk, Dv] product per block is 2 Dk^2 Dv FLOP (4.2 MFLOP at 128): tiny
// next to the segment's forward, so a plain fp32 shared-memory tiling on CUDA cores.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kCT = 64;   // output tile (rows and columns)
constexpr int kCK = 32;   // reduction slice

template <bool TR>
__global__ void __launch_bounds__(256) k_state_compose(int Dk, int Dv, const float* Phi,
                                                       const float* S, const float* R,
                                                       float* out) {
  __shared__ float As[kCK][kCT + 1];  // As[kk][i] = op(Phi)[i0 + i][k0 + kk]
  __shared__ float Bs[kCK][kCT];      // Bs[kk][j] = S[k0 + kk][j0 + j]
  const size_t blk = blockIdx.z;
  const float* P = Phi + blk * (size_t)Dk * Dk;
  const float* Sb = S + blk * (size_t)Dk * Dv;
  const int i0 = blockIdx.y * kCT, j0 = blockIdx.x * kCT;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < Dk; k0 += kCK) {
    for (int e = tid; e < kCK * kCT; e += 256) {
      int i, kk;
      if (TR) {  // op(Phi)[i][kk] = Phi[kk][i]: consecutive threads walk i (a row of Phi)
        kk = e / kCT;
        i = e % kCT;
      } else {   // Phi[i][kk]: consecutive threads walk kk (a row of Phi)
        i = e / kCK;
        kk = e % kCK;
      }
      const int gi = i0 + i, gk = k0 + kk;
      float val = 0.f;
      if (gi < Dk && gk < Dk) val = TR ? P[(size_t)gk * Dk + gi] : P[(size_t)gi * Dk + gk];
      As[kk][i] = val;
    }
    for (int e = tid; e < kCK * kCT; e += 256) {
      const int kk = e / kCT, j = e % kCT, gk = k0 + kk, gj = j0 + j;
      Bs[kk][j] = (gk < Dk && gj < Dv) ? Sb[(size_t)gk * Dv + gj] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kCK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[kk][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = Bs[kk][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
  const float* Rb = R ? R + blk * (size_t)Dk * Dv : nullptr;
  float* Ob = out + blk * (size_t)Dk * Dv;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int gi = i0 + ty * 4 + r;
    if (gi >= Dk) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int gj = j0 + tx * 4 + c;
      if (gj >= Dv) continue;
      const size_t at = (size_t)gi * Dv + gj;
      Ob[at] = acc[r][c] + (Rb ? Rb[at] : 0.f);
    }
  }
}

}  // namespace

cudaError_t launch_state_compose(int n, int Dk, int Dv, const float* Phi, const float* S,
                                 const float* R, float* out, bool transpose, cudaStream_t st) {
  const dim3 grid((unsigned)((Dv + kCT - 1) / kCT), (unsigned)((Dk + kCT - 1) / kCT), (unsigned)n);
  profile_pre(st, KID_COMPOSE);
  if (transpose)
    k_state_compose<true><<<grid, 256, 0, st>>>(Dk, Dv, Phi, S, R, out);
  else
    k_state_compose<false><<<grid, 256, 0, st>>>(Dk, Dv, Phi, S, R, out);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
