// gdn_tc_bwd.cu -- tensor-core (tcgen05) backward for bf16 inputs.
//
// k_bwd_state_tc  one CTA per (sequence, value head): reverse walk over the chunks
//                 with the state adjoint dS^T in registers (fp32) and as a bf16
//                 operand tile.  Per chunk:
//                   dDelta^T = scale (dO^T P) + diag-cols(c) (dS^T K^T)
//                   dS^T    <- e^{G_last} dS^T + (scale e^G dO)^T Q - dDelta^T W
//                 and it stores dS (chunk end) and dDelta for the gradient kernel.
// k_bwd_grads_tc  one CTA per (chunk, key head), looping over the value heads of
//                 the key head; dQ_hat and dK_hat of the key head accumulate in
//                 TMEM across the heads (fixed order: bit-reproducible, no
//                 atomics), then the L2-norm backward writes dq, dk.  Per head it
//                 recomputes Delta = U - W S and forms every chunk-level
//                 derivative of the WY form (see gdn_bwd.cu) with tcgen05 MMAs,
//                 plus the gate / sigmoid epilogues.
#include "gdn_tc.cuh"

namespace gdn {

namespace {
constexpr int C = kChunk;
constexpr int kColParts = kTcThreads / 64;   // row blocks of the column sums of a C x C scratch
__device__ __forceinline__ size_t tileCD(int D) { return (size_t)((D + 63) / 64) * 64 * 128; }
}  // namespace

// ---------------------------------------------------------------------------
// The reverse chunk walk of sequence n, value head h on a whole CTA (`sm`: 1024-aligned,
// bwd_state_tc_smem bytes; `tmem`: 512 columns; bars[0..2]: MMA and the two load
// buffers).  In a fused launch (p.bready set) chunk c's flag is published once its dS^T
// and -dDelta tiles have reached global memory.
template <int DK, int DV>   // DV: the value head size when fixed, else 0 (p.Dv)
__device__ void bwd_state_unit(const Params& p, const TmaMaps& maps, int n, int h, uint8_t* sm,
                               uint32_t tmem, uint64_t* bars) {
  const int kh = key_head(p, h);
  int64_t s0, s1;
  int c0, c1;
  if (!seq_info(p, n, &s0, &s1, &c0, &c1)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, n);
    return;
  }
  constexpr int NKC = (DK + 16 * kGroups - 1) / (16 * kGroups);   // dS^T pieces per thread
  const int Dv = DV > 0 ? DV : p.Dv, MV = Dv < 64 ? 64 : Dv;
  const int tid = threadIdx.x, grp = col_group();
  constexpr int NKF = DK < 64 ? 64 : DK;        // N of products read Q / W MN-major
  const uint32_t bK = (uint32_t)tileCD(DK), bP = 8192, bG = C * 4;
  const int nbv = (Dv + 63) / 64;
  const uint32_t bO = (uint32_t)nbv * 8192;                  // natural dO tile [C][Dv]
  const uint32_t bSt = tc::sw128_bytes(MV, DK);              // dS^T tile
  const uint32_t bD = tc::sw128_bytes(C, MV);
  uint8_t* tdSt = sm;                                        // [MV][DK] dS^T
  uint8_t* tmD = tdSt + bSt;                                 // [C][MV] -dDelta (token rows)
  uint8_t* buf0 = tmD + bD;
  const uint32_t bufsz = bO + 3 * bK + bP + 1024;
  float* ev = (float*)(buf0 + 2 * bufsz);
  float* cv = ev + C;
  // per stage buffer: the natural tiles of dO (TMA), K, P, Q (scaled in place to
  // scale e^G Q), W and the gates G; every transposed operand is read MN-major
  auto sdO = [&](int b) { return buf0 + b * bufsz; };
  auto tK = [&](int b) { return buf0 + b * bufsz + bO; };
  auto tP = [&](int b) { return buf0 + b * bufsz + bO + bK; };
  auto tQ = [&](int b) { return buf0 + b * bufsz + bO + bK + bP; };
  auto tW = [&](int b) { return buf0 + b * bufsz + bO + 2 * bK + bP; };
  auto sG = [&](int b) { return (const float*)(buf0 + b * bufsz + bO + 3 * bK + bP); };

  for (int i = tid; i < (int)(bSt + bD) / 16; i += kTcThreads)
    ((uint4*)tdSt)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // fused launch: chunks whose tiles are in global memory are published (thread 0;
  // the walk goes down, so every chunk >= published is)
  int published = c1;
  auto publish_down_to = [&](int cc) {
    if (published > cc) {
      publish_flags(p.bready + ((size_t)cc * p.Hv + h), (size_t)p.Hv, published - cc);
      published = cc;
    }
  };
  // TMEM: dS^T update (rows v) @0; in token rows (M = 64): P^T dO @128, K dS @256
  const uint32_t tA3 = tmem, tA1 = tmem + 128, tA2 = tmem + 256;
  uint32_t mphase = 0, lph[2] = {0, 0};
  const int vrow = acc_row(MV);
  const bool vok = vrow >= 0 && vrow < Dv;
  const size_t SZ = (size_t)DK * Dv;

  float dS[NKC][16];
#pragma unroll
  for (int i = 0; i < NKC; ++i)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int k = grp * 16 + 16 * kGroups * i + j;
      dS[i][j] = (vok && k < DK && p.dS_T) ? p.dS_T[((size_t)n * p.Hv + h) * SZ + (size_t)k * Dv + vrow] : 0.f;
    }
#pragma unroll
  for (int i = 0; i < NKC; ++i)
    if (grp * 16 + 16 * kGroups * i < DK && vok)
      tile_put16(tdSt, MV, vrow, grp * 16 + 16 * kGroups * i, dS[i]);
  tc::fence_async_smem();

  auto issue_load = [&](int cc, int b) {
    uint64_t* lb = &bars[1 + b];
    const size_t chh = (size_t)cc * p.Hv + h, ckk = (size_t)cc * p.Hk + kh;
    tc::mbar_arrive_expect_tx(lb, bO + 3 * bK + bP + bG);
    for (int b2 = 0; b2 < nbv; ++b2)
      tc::tma_load_2d(sdO(b) + b2 * 8192, &maps.dO, h * Dv + 64 * b2,
                      (int)(s0 + (int64_t)(cc - c0) * C), lb);
    tc::bulk_g2s(tK(b), p.Ksw + ckk * bK, bK, lb);
    tc::bulk_g2s(tP(b), p.Psw + chh * bP, bP, lb);
    tc::bulk_g2s(tQ(b), p.Qsw + ckk * bK, bK, lb);
    tc::bulk_g2s(tW(b), p.Wsw + chh * bK, bK, lb);
    tc::bulk_g2s((void*)sG(b), p.G + chh * C, bG, lb);
  };
  if (tid == 0 && c1 > c0) issue_load(c1 - 1, 0);

  bool ok = true;
  for (int c = c1 - 1; c >= c0 && ok; --c) {
    const int i = c1 - 1 - c, b = i & 1;
    const int64_t t0 = s0 + (int64_t)(c - c0) * C;
    const int len = (int)((s1 - t0) < C ? (s1 - t0) : C);
    const size_t ch = (size_t)c * p.Hv + h;
    const bool lok = tc::mbar_wait(&bars[1 + b], lph[b]);
    lph[b] ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
      ok = false;
      break;
    }
    // the next chunk's tiles into the other buffer (every read of it by the last chunk
    // is done, its in-place writes fenced), by another thread than the products' issuer
    if (tid == 32 && c - 1 >= c0) issue_load(c - 1, b ^ 1);
    if (tid == 0) {
      // every fourth chunk (every chunk at first, when gradient units are waiting for
      // the walk), before this chunk's first store: all but the last two store groups
      // (the previous chunk's) have landed, so the chunks down to c + 2 are published
      // (later the gradient units trail the walk; waiting only for old stores keeps the
      // wait short)
      if (p.bready && i > 1 && (i < 8 || (i & 3) == 0)) {
        tc::bulk_wait<2>();
        publish_down_to(c + 2);
      }
      // state adjoint at the end of this chunk: the dS^T tile, by one bulk store
      tc::bulk_s2g(p.dSb + ch * bSt, tdSt, bSt);
      tc::bulk_commit();
    }
    const float* G = sG(b);
    if (tid < C) {
      ev[tid] = expf(G[tid]);
      cv[tid] = tid < len ? expf(G[len - 1] - G[tid]) : 0.f;
    }
    __syncthreads();
    // rows of the dO tile past the chunk (another sequence's tokens) read as zero
    if (len < C)
      for (int idx = tid; idx < nbv * (C - len) * 8; idx += kTcThreads) {
        const int b2 = idx / ((C - len) * 8), rem = idx % ((C - len) * 8);
        ((uint4*)(sdO(b) + b2 * 8192 + (len + rem / 8) * 128))[rem % 8] = make_uint4(0, 0, 0, 0);
      }
    // scale e^G Q in place: row r of the natural Q tile times scale e^{G_r}
    for (int idx = tid; idx < C * (DK / 8); idx += kTcThreads) {
      const int r = idx % C, k8 = (idx / C) * 8;
      uint4* at = (uint4*)(tQ(b) + tc::sw128_offset(r, k8, C));
      const uint4 raw = *at;
      const __nv_bfloat162* e = (const __nv_bfloat162*)&raw;
      const float sc = p.scale * ev[r];
      __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(e[q]);
        pk[q] = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      }
      *at = *(const uint4*)pk;
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      tc::bulk_wait_read<1>();   // last chunk's dDelta store has read its tile
      // token rows s: P^T dO (both operands MN-major: P^T from the natural P tile, dO
      // from the natural dO boxes, 8 KB apart) and K dS (B = the dS^T tile)
      tc::mma_tile_x(tA1, tc::smem_u32(tP(b)), true, 8192u, 64, tc::smem_u32(sdO(b)), true,
                     8192u, MV, C, 0u);
      tc::mma_tile_p(tA2, tc::smem_u32(tK(b)), 8192u, 64, tc::smem_u32(tdSt), (uint32_t)MV * 128u,
                     Dv, DK, 0u);
      // rows v: dO^T (scale e^G Q), dO^T read MN-major
      tc::mma_tile_x(tA3, tc::smem_u32(sdO(b)), true, 8192u, MV, tc::smem_u32(tQ(b)), true,
                     8192u, NKF, C, 0u);
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // dDelta = scale P^T dO + diag(c) K dS, stored negated in token rows (the A
    // operand of the update below, read MN-major, and the gradient kernel's tile)
    {
      // M = 64 accumulators, two 16-column pieces per load (x2_row / x2_half)
      const int s = x2_row();
      for (int c0 = grp * 16; c0 < Dv; c0 += 32 * kGroups) {
        float a1[16], a2[16];
        tc::tmem_ld16_x2<16 * kGroups>(tA1 + lane_quarter() + c0, a1);
        tc::tmem_ld16_x2<16 * kGroups>(tA2 + lane_quarter() + c0, a2);
        tc::tmem_ld_wait();
        const int col = c0 + x2_half() * 16 * kGroups;
        if (col < Dv) {
          float md[16];
          if (s < len) {
            const float cs = cv[s];
#pragma unroll
            for (int j = 0; j < 16; ++j) md[j] = -fmaf(p.scale, a1[j], cs * a2[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) md[j] = 0.f;
          }
          tile_put16(tmD, C, s, col, md);
        }
      }
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      tc::mma_tile_x(tA3, tc::smem_u32(tmD), true, 8192u, MV, tc::smem_u32(tW(b)), true, 8192u,
                     NKF, C, 1u);
      tc::bulk_wait_read<0>();   // the dS^T store has read its tile: the update may rewrite it
      tc::bulk_s2g(p.dDb + ch * bD, tmD, bD);
      tc::bulk_commit();
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    const float eC = expf(G[len - 1]);
#pragma unroll
    for (int ii = 0; ii < NKC; ++ii) {
      const int col0 = grp * 16 + 16 * kGroups * ii;
      if (col0 < DK) {
        float x[16];
        tc::tmem_ld16(tA3 + lane_quarter() + col0, x);
        tc::tmem_ld_wait();
        if (vok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) dS[ii][j] = fmaf(eC, dS[ii][j], x[j]);
          tile_put16(tdSt, MV, vrow, col0, dS[ii]);
        }
      }
    }
    tc::fence_async_smem();
  }
  if (ok && p.dS0 && vok)
#pragma unroll
    for (int ii = 0; ii < NKC; ++ii)
      if (grp * 16 + 16 * kGroups * ii < DK)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          p.dS0[((size_t)n * p.Hv + h) * SZ + (size_t)(grp * 16 + 16 * kGroups * ii + j) * Dv +
                vrow] = dS[ii][j];
  if (tid == 0) {
    tc::bulk_wait<0>();
    // the rest (also after an error: consumers then read what there is, the status
    // word already holds the error)
    if (p.bready) publish_down_to(c0);
  }
  __syncthreads();
}

template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_bwd_state_tc(Params p,
                                                               const __grid_constant__ TmaMaps maps) {
  if (kept_operands_missing(p)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  cta_setup(ctl, 4, 512);
  bwd_state_unit<DK, DV>(p, maps, blockIdx.x, blockIdx.y, base + kCtlBytes, ctl->tmem, ctl->bar);
  cta_teardown(ctl, 512);
}

// ---------------------------------------------------------------------------
// Shared-memory plan of k_bwd_grads_tc (bytes for Dk = Dv = 128; phases A-E of one
// value head reuse the regions):
//   R1 65K  A: S^T [Dv][Dk] (also read MN-major as S) | B: Delta^T, c Delta^T [Dv][C],
//           dW [C][Dk]
//           C-E: dPE, dT, H [C][C] (over Delta / c*Delta)
//           A-E, from 48K: K K^T of the key head, fp32 [C][C + 4] (whole CTA)
//   R2 32K  A-B: [dO; -dDelta] [128][Dv]  | B-E: fp32 [C][C] scratch
//   R3 48K  A: W [C][Dk], scale e^G dO [C][Dv], U^T [Dv][C] | B: dS^T [Dv][Dk], P [C][C]
//           C-E: -dDelta^T [Dv][C], T, T diag(b e^G), Y [C][C]
//   R4 32K  B-C: V [C][Dv], -e^G K [C][Dk]
//   R5 32K  K, Q [C][Dk] of the key head (whole CTA)
// Every transposed operand (T^T, dW^T, dPE^T, dT^T, K^T, Q^T, S, dS) is a natural
// tile read MN-major.
// TMEM (512 columns): dQ_hat @0, dK_hat @128 (M = 64 accumulators), scratch @256.
// One (chunk c, key head kh) gradient unit on a whole CTA (`sm`: 1024-aligned,
// grads_tc_smem bytes; `tmem`: 512 columns; bars[0] / bars[1]: MMA and loads with
// their running phases).  In a fused launch (p.bready set) it first waits until the
// reverse walks of the key head's value heads have published chunk c.
// The bf16 S^T tiles of the chunk-start states the backward reads, if there are any: the
// saved states (GDN_FLAG_BF16_SAVED_STATES) or the copy kept by the forward of a
// training step; null when the fp32 saved states are converted instead.
__device__ __forceinline__ const uint8_t* st_tile_source(const Params& p) {
  return p.bf16_states ? (const uint8_t*)p.saved_in : (p.reuse ? p.Stb : nullptr);
}

// Thread 0: the fp32 chunk-start states of unit (c, kh)'s value heads into the L2 (heads
// from `first` on), so that their conversion to the S^T tile does not wait on HBM.
__device__ __forceinline__ void prefetch_unit_states(const Params& p, int c, int kh, int first) {
  if (st_tile_source(p) || c < 0) return;
  const uint32_t bytes = (uint32_t)p.Dk * p.Dv * 4u;
  for (int hh = first; hh < p.r; ++hh) {
    const float* s = p.saved_in + ((size_t)c * p.Hv + value_head(p, kh, hh)) * (size_t)p.Dk * p.Dv;
    for (uint32_t off = 0; off < bytes; off += 16384u)
      tc::bulk_prefetch_l2((const uint8_t*)s + off, bytes - off < 16384u ? bytes - off : 16384u);
  }
}

template <int DK, int DV>   // DV: the value head size when fixed, else 0 (p.Dv)
__device__ void grads_unit(const Params& p, const TmaMaps& maps, int c, int kh, uint8_t* sm,
                           uint32_t tmem, uint64_t* bars, uint32_t& mphase, uint32_t& lphase,
                           int next_c = -1, int next_kh = 0) {
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  constexpr int Dk = DK;   // the head sizes p.Dk, p.Dv, fixed by the instantiation where it can
  const int Dv = DV > 0 ? DV : p.Dv;
  const int tid = threadIdx.x, warp = tid >> 5, grp = col_group();
  const uint32_t sCK = tc::sw128_bytes(C, Dk), sCV = tc::sw128_bytes(C, Dv);
  const uint32_t sCC = 8192;
  // tiles handed over by the state kernels: S^T and dS^T [MV][Dk], -dDelta^T [MV][C],
  // -dDelta [C][MV] (MV = Dv rounded up to 64); MMAs whose N is Dk read S / dS
  // MN-major with N rounded up to 64 (the tiles' padding columns are zero)
  const int MV = Dv < 64 ? 64 : Dv;
  constexpr int NK = Dk < 64 ? 64 : Dk;
  const uint32_t bSt = tc::sw128_bytes(MV, Dk), sVC = (uint32_t)MV * 128;
  uint8_t* R1 = sm;
  uint8_t* R2 = R1 + 66560;
  uint8_t* R3 = R2 + 32768;
  uint8_t* R4 = R3 + 49152;
  uint8_t* R5 = R4 + 32768;
  // R1
  uint8_t* tSt = R1;                               // [MV][Dk] S^T (K-major), S (MN-major)
  uint8_t* tDl = R1;                               // [Dv][C] Delta^T (read MN-major as Delta)
  uint8_t* tDlc = R1 + 16384;                      // [Dv][C] Delta^T diag(c)
  uint8_t* tdW = R1 + 32768;                       // [C][Dk]
  uint8_t* tdPE = R1;                              // [C][C]
  uint8_t* tdT = R1 + 16384;                       // [C][C]
  uint8_t* tH = R1 + 24576;                        // [C][C] H = dA b_r E (strictly lower)
  float* sKK = (float*)(R1 + 49152);               // [C][KKL] fp32 K K^T (padded rows)
  constexpr int KKL = C + 4;
  // per-row partial sums of the kGroups column groups, added in a fixed order
  auto rsum_g = [&](const float* a, int t) {
    float v = a[t];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) v += a[g * C + t];
    return v;
  };
  // R2
  uint8_t* tA2 = R2;                               // [128][Dv]: rows 0-63 dO, 64-127 -dDelta
  float* X = (float*)R2;                           // [C][C + 1] fp32 scratch (padded rows)
  constexpr int XL = C + 1;
  // R3
  uint8_t* tW = R3;                                // [C][Dk]
  uint8_t* tdOe = R3 + 16384;                      // [C][Dv]
  uint8_t* sU = R3 + 32768;                        // [Dv][C] SW128 tile of U^T
  uint8_t* tdS = R3;                               // [MV][Dk] dS^T (read MN-major as dS)
  uint8_t* tP = R3 + 32768;                        // [C][C]
  uint8_t* tdDt = R3;                              // [C][MV] -dDelta (read MN-major)
  uint8_t* tT = R3 + 16384;                        // [C][C] T
  uint8_t* tTW = R3 + 24576;                       // [C][C] T diag(b e^G)
  uint8_t* tY = R3 + 40960;
  // R4
  uint8_t* tV = R4;                                // [C][Dv]
  uint8_t* tKe = R4 + 16384;                       // [C][Dk] -e^G K
  // R5
  uint8_t* tK = R5;                                // [C][Dk]
  uint8_t* tQ = R5 + 16384;                        // [C][Dk]
  float* vec = (float*)(R5 + 32768);
  float* gv = vec;            // G
  float* ev = gv + C;         // e^G
  float* cv = ev + C;         // e^{G_last - G}
  float* bv = cv + C;         // beta
  float* dG = bv + C;         // dL/dG
  float* db = dG + C;         // dL/d beta
  float* xa = db + C;         // alpha + dt_bias of the chunk's tokens
  float* part = xa + C;       // [kGroups][C] per-group partial row sums
  float* rowp = part + kGroups * C;  // [kGroups][C] per-group partial row sums
  float* colp = rowp + kGroups * C;  // [kColParts][C] partial column sums
  float* invn = colp + kColParts * C;  // [2][C] |q|, |k| of the chunk's tokens
  float* al = invn + 2 * C;   // a_log of the value head, one copy per token slot
  float* stg = al + C;        // [2][5][C] next value head's G, beta, alpha, dt_bias, a_log
  float* red = stg + 10 * C;  // [kTcThreads / 32]

  const uint32_t tdQ = tmem, tdK = tmem + 128, tmp = tmem + 256;
  const size_t ckk = (size_t)c * p.Hk + kh;
  bool ok = true;

  // Phase A's tiles of value head h: S^T, W, U^T (bulk copies), dO rows into the
  // [dO; -dDelta] tile and V rows (TMA) need nothing from the reverse walks; the
  // -dDelta rows (bulk) are the walk's and wait for its flag.  All land in one phase
  // of bars[1] of phase_a_bytes.
  const int nbv = (Dv + 63) / 64;
  // the S^T tile is a bulk copy of a bf16 state tile: the saved state itself
  // (GDN_FLAG_BF16_SAVED_STATES) or the copy a keeping forward left for a reusing
  // backward; otherwise the whole CTA converts the fp32 saved state (load_state_f32)
  const uint8_t* st_tiles = st_tile_source(p);
  const uint32_t phase_a_bytes =
      sCK + (uint32_t)Dv * C * 2 + 3u * nbv * 8192u + (st_tiles ? bSt : 0u);
  auto issue_phase_a_inputs = [&](int h) {
    const size_t ch = (size_t)c * p.Hv + h;
    if (st_tiles) tc::bulk_g2s(tSt, st_tiles + ch * bSt, bSt, &bars[1]);
    tc::bulk_g2s(tW, p.Wsw + ch * sCK, sCK, &bars[1]);
    tc::bulk_g2s(sU, p.Utb + ch * Dv * C, (uint32_t)Dv * C * 2, &bars[1]);
    for (int b = 0; b < nbv; ++b) {
      tc::tma_load_2d(tA2 + b * 16384, &maps.dO, h * Dv + 64 * b, (int)t0, &bars[1]);
      tc::tma_load_2d(tV + b * 8192, &maps.v, h * Dv + 64 * b, (int)t0, &bars[1]);
    }
  };
  auto issue_phase_a_walk = [&](int h) {
    const size_t ch = (size_t)c * p.Hv + h;
    for (int b = 0; b < nbv; ++b)
      tc::bulk_g2s(tA2 + b * 16384 + 8192, p.dDb + ch * sCV + b * 8192, 8192, &bars[1]);
  };
  // G, beta, alpha, dt_bias and a_log of value head h into staging buffer h & 1 (token
  // slot tid; the alpha rows past the chunk are not read)
  auto prefetch_vectors = [&](int hh) {
    if (tid < C) {
      const int h = value_head(p, kh, hh);
      const size_t ch = (size_t)c * p.Hv + h;
      float* sg = stg + (hh & 1) * 5 * C;
      tc::cp_async4(sg + tid, p.G + ch * C + tid);
      tc::cp_async4(sg + C + tid, p.b + ch * C + tid);
      if (tid < len) tc::cp_async4(sg + 2 * C + tid, p.alpha + (t0 + tid) * p.alpha_ld + h);
      tc::cp_async4(sg + 3 * C + tid, p.dt_bias + h);
      tc::cp_async4(sg + 4 * C + tid, p.a_log + h);
    }
  };

  // The chunk-start state of value head h as the bf16 S^T tile tSt (rows v, columns k),
  // converted by the whole CTA from the fp32 saved state.  Items (k pair kp, block of 8
  // value columns v8), consecutive lanes on consecutive kp so that the 4-byte (k, k + 1)
  // stores of a warp fall in distinct banks.  The tile then also goes to the workspace
  // (Stb), from where phase B reads it back for <S, dS> exactly as it reads a kept tile.
  const int nkp = Dk / 2, n_items = (Dk / 2) * (Dv / 8);
  constexpr int kItems = 2;   // items per thread: Dk * Dv / 16 <= 2 * kTcThreads
  auto load_state_f32 = [&](int h) {
    const size_t ch = (size_t)c * p.Hv + h;
    const float* Sf = p.saved_in + ch * (size_t)Dk * Dv;
    if (Dv < 64 || Dk < 64) {   // the tile's padding rows / columns read as zero
      for (int i = tid; i < (int)bSt / 16; i += kTcThreads) ((uint4*)tSt)[i] = make_uint4(0, 0, 0, 0);
      __syncthreads();
    }
    float4 x[kItems][4];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads, kp = i % nkp, v0 = (i / nkp) * 8;
      if (i < n_items) {
        const float* r0 = Sf + (size_t)(2 * kp) * Dv + v0;
        x[u][0] = *(const float4*)r0;
        x[u][1] = *(const float4*)(r0 + 4);
        x[u][2] = *(const float4*)(r0 + Dv);
        x[u][3] = *(const float4*)(r0 + Dv + 4);
      }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads, kp = i % nkp, v0 = (i / nkp) * 8;
      if (i < n_items) {
        const float a[8] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w,
                            x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
        const float b[8] = {x[u][2].x, x[u][2].y, x[u][2].z, x[u][2].w,
                            x[u][3].x, x[u][3].y, x[u][3].z, x[u][3].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          __nv_bfloat162 pr = __floats2bfloat162_rn(a[j], b[j]);
          *(__nv_bfloat162*)(tSt + tc::sw128_offset(v0 + j, 2 * kp, MV)) = pr;
        }
      }
    }
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::bulk_s2g(p.Stb + ch * bSt, tSt, bSt);
      tc::bulk_commit();
    }
  };

  // fp32 states: this unit's later value heads and the next unit's into the L2 (the
  // first head's conversion follows at once)
  if (tid == 0) {
    prefetch_unit_states(p, c, kh, 1);
    prefetch_unit_states(p, next_c, next_kh, 0);
  }
  // K, Q of the key head and the first value head's phase-A tiles in one phase of
  // bars[1]; the copies that need no walk start before the flags are read
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&bars[1], 2 * sCK + phase_a_bytes);
    tc::bulk_g2s(tK, p.Ksw + ckk * sCK, sCK, &bars[1]);
    tc::bulk_g2s(tQ, p.Qsw + ckk * sCK, sCK, &bars[1]);
    issue_phase_a_inputs(value_head(p, kh, 0));
  }
  // K K^T of the key head into padded rows (conflict-free row reads in epilogue D),
  // the norms for the L2 backward at the end and the first head's vectors
  for (int i = tid; i < C * C / 4; i += kTcThreads)
    tc::cp_async16(sKK + (i / (C / 4)) * KKL + (i % (C / 4)) * 4, p.KKf + ckk * C * C + i * 4);
  if (tid < 2 * C) tc::cp_async4(invn + tid, (tid < C ? p.nq : p.nk) + ckk * C + (tid & (C - 1)));
  prefetch_vectors(0);
  // fused launch: this chunk's dS^T / -dDelta tiles of every value head of the group
  // (one thread per value head)
  if (p.bready) {
    for (int hh = tid; hh < p.r; hh += kTcThreads)
      if (!wait_flag(p.bready + (size_t)c * p.Hv + value_head(p, kh, hh)))
        set_status(p.status, GDN_ERR_TIMEOUT, c);
    __syncthreads();
  }
  if (tid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    issue_phase_a_walk(value_head(p, kh, 0));
  }
  for (int hh = 0; hh < p.r && ok; ++hh) {
    const int h = value_head(p, kh, hh);
    const size_t ch = (size_t)c * p.Hv + h;
    const uint32_t acc_first = hh > 0 ? 1u : 0u;
    // S^T tile in global memory for <S, dS>: the kept / saved tile, or the converted one
    const uint8_t* Sg = (st_tiles ? st_tiles : p.Stb) + ch * bSt;
    // this head's vectors (prefetched), then the next head's prefetch
    tc::cp_async_wait_all();
    if (tid < C) {
      const float* sg = stg + (hh & 1) * 5 * C;
      gv[tid] = sg[tid];
      bv[tid] = sg[C + tid];
      xa[tid] = tid < len ? sg[2 * C + tid] + sg[3 * C + tid] : 0.f;
      al[tid] = sg[4 * C + tid];
      dG[tid] = 0.f;
      db[tid] = 0.f;
    }
    if (hh + 1 < p.r) prefetch_vectors(hh + 1);
    // phase A's tiles were issued at the start of the unit (first head) or when the
    // previous head's last product finished
    __syncthreads();
    if (tid < C) {
      ev[tid] = expf(gv[tid]);
      cv[tid] = tid < len ? expf(gv[len - 1] - gv[tid]) : 0.f;
    }
    __syncthreads();
    // ---- phase A: S^T, [dO; -dDelta], scale e^G dO
    if (!st_tiles) load_state_f32(h);
    {
      const bool lok = tc::mbar_wait(&bars[1], lphase);
      lphase ^= 1u;
      if (__syncthreads_or(lok ? 0 : 1)) {
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
        ok = false;
        break;
      }
    }
    // scale e^G dO (rows past the chunk zero) from the dO rows of the [dO; dDelta] tile
    for (int idx = tid; idx < C * (Dv / 8); idx += kTcThreads) {
      const int r = idx % C, c8 = (idx / C) * 8;
      const uint4 raw = *(const uint4*)(tA2 + tc::sw128_offset(r, c8, 128));
      const __nv_bfloat16* e = (const __nv_bfloat16*)&raw;
      const float sc = r < len ? p.scale * ev[r] : 0.f;
      __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        pk[q] = __floats2bfloat162_rn(__bfloat162float(e[2 * q]) * sc, __bfloat162float(e[2 * q + 1]) * sc);
      *(uint4*)(tdOe + tc::sw128_offset(r, c8, C)) = *(const uint4*)pk;
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      // a converted tile's store to the workspace has read tSt before epilogue A reuses it
      if (!st_tiles) tc::bulk_wait_read<0>();
      tc::mma_tile_p(tmp, tc::smem_u32(tSt), sVC, MV, tc::smem_u32(tW), 64u * 128u, C, Dk,
                     0u);                                                                // S^T W^T
      tc::mma_tile_x(tmp + 128, tc::smem_u32(tA2), false, 128u * 128u, 128, tc::smem_u32(tSt),
                     true, sVC, NK, Dv, 0u);                                             // [dO;-dD] S^T
      tc::mma_tile_x(tdQ, tc::smem_u32(tdOe), false, 64u * 128u, 64, tc::smem_u32(tSt), true,
                     sVC, NK, Dv, acc_first);                                            // dQ += s e^G dO S^T
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // the dS^T tile lands over W and scale e^G dO (read by the products above) while
    // epilogue A runs; P follows once epilogue A has read U^T
    if (tid == 0) {
      tc::mbar_expect_tx(&bars[1], bSt);
      tc::bulk_g2s(tdS, p.dSb + ch * bSt, bSt, &bars[1]);
    }
    // epilogue A: Delta^T = U^T - S^T W^T; dG += scale e^G (Q . dO S^T); dW = -dDelta S^T
    // (the lower half of the stacked product)
    if (tid < kGroups * C) part[tid] = 0.f;
    __syncthreads();
    acc_walk(tmp, MV, C, Dv, [&](int v, int col0, const float* x) {
      float d[16], dc[16];
      tile_get16(sU, Dv, v, col0, d);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        d[j] -= x[j];
        dc[j] = d[j] * cv[col0 + j];
      }
      tile_put16(tDl, Dv, v, col0, d);
      tile_put16(tDlc, Dv, v, col0, dc);
    });
    {
      const int row = acc_row(128);
      float rs = 0.f;
      for (int q = grp; q * 16 < Dk; q += kGroups) {
        float x[16];
        tc::tmem_ld16(tmp + 128 + lane_quarter() + q * 16, x);
        tc::tmem_ld_wait();
        if (row < C) {
          float qv[16];
          tile_get16(tQ, C, row, q * 16, qv);
#pragma unroll
          for (int j = 0; j < 16; ++j) rs = fmaf(qv[j], x[j], rs);
        } else {
          tile_put16(tdW, C, row - C, q * 16, x);
        }
      }
      if (row < C) part[grp * C + row] = rs;
    }
    // phase B's products that need no dS^T (dO Delta^T and -dDelta V^T) are issued now,
    // once epilogue A's tiles and TMEM reads are done, and run under the -e^G K pass and
    // the dS^T load; the rest follow behind them and one commit covers all five
    const uint32_t dvp = (uint32_t)Dv * 128u;   // Delta^T tiles read MN-major
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_tile_x(tmp + 128, tc::smem_u32(tA2), false, 128u * 128u, 64, tc::smem_u32(tDl), true,
                     dvp, C, Dv, 0u);                                                    // dO Delta^T
      tc::mma_tile_p(tmp + 192, tc::smem_u32(tA2) + 64u * 128u, 128u * 128u, 64,
                     tc::smem_u32(tV), (uint32_t)C * 128u, C, Dv, 0u);                  // -dDelta V^T
    }
    if (tid < C) dG[tid] += p.scale * ev[tid] * rsum_g(part, tid);
    // ---- phase B: dS tile, P tile (bulk), e^G K from K^T, <S, dS>
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(&bars[1], sCC);
      tc::bulk_g2s(tP, p.Psw + ch * sCC, sCC, &bars[1]);
    }
    // S^T again, from global memory (L2), for <S, dS>: the shared copy is gone.  A tile
    // converted here was stored by this unit's bulk copy: it has landed and is visible
    // to the generic loads once thread 0 has waited for it, fenced and met the others
    if (!st_tiles) {
      if (tid == 0) {
        tc::bulk_wait<0>();
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncthreads();
    }
    constexpr int kSraw = 32768 / 16 / kTcThreads;   // 16-byte pieces per thread (32 KB tile max)
    uint4 sraw[kSraw];
#pragma unroll
    for (int u = 0; u < kSraw; ++u) {
      const uint32_t i = tid + u * kTcThreads;
      sraw[u] = i < bSt / 16 ? ((const uint4*)Sg)[i] : make_uint4(0, 0, 0, 0);
    }
    for (int idx = tid; idx < C * (Dk / 8); idx += kTcThreads) {
      const int s = idx % C, k8 = (idx / C) * 8;
      const uint32_t off = tc::sw128_offset(s, k8, C);
      const uint4 raw = *(const uint4*)(tK + off);
      const __nv_bfloat162* e = (const __nv_bfloat162*)&raw;
      const float sc = -ev[s];
      __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(e[u]);
        pk[u] = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      }
      *(uint4*)(tKe + off) = *(const uint4*)pk;
    }
    {
      const bool lok = tc::mbar_wait(&bars[1], lphase);
      lphase ^= 1u;
      if (__syncthreads_or(lok ? 0 : 1)) {
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
        ok = false;
        break;
      }
    }
    {
      // <S, dS>: the S^T and dS^T tiles share one layout (zero padding included), so
      // the dot product runs over them flat
      float sds = 0.f;
#pragma unroll
      for (int u = 0; u < kSraw; ++u) {
        const uint32_t i = tid + u * kTcThreads;
        if (i < bSt / 16) {
          const uint4 raw = ((const uint4*)tdS)[i];
          const __nv_bfloat162* a = (const __nv_bfloat162*)&sraw[u];
          const __nv_bfloat162* d = (const __nv_bfloat162*)&raw;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 fa = __bfloat1622float2(a[q]), fd = __bfloat1622float2(d[q]);
            sds = fmaf(fa.x, fd.x, fmaf(fa.y, fd.y, sds));
          }
        }
      }
      sds = warp_sum(sds);
      if ((tid & 31) == 0) red[warp] = sds;
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      tc::mma_tile_x(tmp, tc::smem_u32(tDlc), true, dvp, 64, tc::smem_u32(tdS), true, sVC, NK, Dv,
                     0u);                                                                // c Delta dS^T
      tc::mma_tile_x(tdK, tc::smem_u32(tDlc), true, dvp, 64, tc::smem_u32(tdS), true, sVC, NK, Dv,
                     acc_first);                                                         // dK +=
      tc::mma_tile(tmp + 192, tc::smem_u32(tdW), 64, tc::smem_u32(tKe), C, Dk, 1u);     // - dW (e^G K)^T
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // phase C's tiles land in the dS^T space (free now) while epilogue B runs
    if (tid == 0) {
      const uint8_t* tb = p.Tb + ch * 2 * sCC;
      tc::mbar_arrive_expect_tx(&bars[1], sCV + 2 * sCC);
      tc::bulk_g2s(tdDt, p.dDb + ch * sCV, sCV, &bars[1]);
      tc::bulk_g2s(tT, tb, sCC, &bars[1]);
      tc::bulk_g2s(tTW, tb + sCC, sCC, &bars[1]);
    }
    // epilogue B
    {
      float rs = 0.f;
      acc_walk64(tmp, Dk, C, [&](int r, int col0, const float* x) {
        float kv[16];
        tile_get16(tK, C, r, col0, kv);
#pragma unroll
        for (int j = 0; j < 16; ++j) rs = fmaf(kv[j], x[j], rs);
      });
      rs = x2_pair_sum(rs);
      if (x2_half() == 0) part[grp * C + x2_row()] = rs;  // c_s * dc_s
    }
    {
      // dO Delta^T @128 and the dT terms @192, 8 columns per thread
      float rsum = 0.f;
      {
        const int r = x2_row(), s0 = grp * 16 + 8 * x2_half();
        float x[8], y[8];
        tc::tmem_ld8_x2<8>(tmp + 128 + lane_quarter() + grp * 16, x);
        tc::tmem_ld8_x2<8>(tmp + 192 + lane_quarter() + grp * 16, y);
        tc::tmem_ld_wait();
        if (s0 < C) {
          float pv[8], pe[8], dt[8];
          tile_get8(tP, C, r, s0, pv);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int s = s0 + j;
            const float dP = (s <= r && r < len) ? p.scale * x[j] : 0.f;
            const float E = s <= r ? expf(gv[r] - gv[s]) : 0.f;
            const float xp = dP * pv[j];
            X[r * XL + s] = xp;
            rsum += xp;
            pe[j] = dP * E;
            dt[j] = -bv[s] * y[j];   // dT[r][s] = b_s (dDelta V^T + dW (e^G K)^T)[r][s]
          }
          tile_put8(tdPE, C, r, s0, pe);
          tile_put8(tdT, C, r, s0, dt);
        }
      }
      rsum = x2_pair_sum(rsum);
      if (x2_half() == 0) rowp[grp * C + x2_row()] = rsum;
    }
    __syncthreads();
    {
      // column sums of X in four quarters of rows
      const int t = tid & (C - 1), qd = tid / C;
      constexpr int rows = C / kColParts;
      float cs = 0.f;
#pragma unroll 4
      for (int r = qd * rows; r < qd * rows + rows; ++r) cs += X[r * XL + t];
      colp[qd * C + t] = cs;
    }
    __syncthreads();
    if (tid < C) {
      const int t = tid, l = tid & 31;
      float csum = 0.f;
#pragma unroll
      for (int g = 0; g < kColParts; ++g) csum += colp[g * C + t];
      float upd = rsum_g(rowp, t) - csum - rsum_g(part, t);
      // the last token takes e^{G_last} <S, dS> + sum_s c_s dc_s: both warps reduce all
      // rows and all warp partials in the same order
      float sc = rsum_g(part, l) + rsum_g(part, l + 32);
      float tot = l < kTcThreads / 32 ? red[l] : 0.f;
      sc = warp_sum(sc);
      tot = warp_sum(tot);
      if (t == len - 1) upd += expf(gv[len - 1]) * tot + sc;
      dG[t] += upd;
    }
    // ---- phase C: -dDelta^T, T, T diag(b e^G) (issued after the MMAs of phase B)
    {
      const bool lok = tc::mbar_wait(&bars[1], lphase);
      lphase ^= 1u;
      if (__syncthreads_or(lok ? 0 : 1)) {
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
        ok = false;
        break;
      }
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      const uint32_t T_ = tc::smem_u32(tT);
      tc::mma_tile_x(tdQ, tc::smem_u32(tdPE), false, sCC, 64, tc::smem_u32(tK), true, 8192u, NK,
                     C, 1u);                                                               // dQ += dPE K
      tc::mma_tile_x(tdK, tc::smem_u32(tdPE), true, sCC, 64, tc::smem_u32(tQ), true, 8192u, NK,
                     C, 1u);                                                               // dK += dPE^T Q
      tc::mma_tile_x(tmp, T_, true, sCC, 64, tc::smem_u32(tdDt), true, 8192u, MV, C, 0u); // -dBv = T^T (-dD)
      tc::mma_tile_x(tmp + 128, T_, true, sCC, 64, tc::smem_u32(tdT), true, sCC, C, C, 0u); // Y = T^T dT
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // epilogue C: dv = b dBv, db += rowsum(dBv * V), Y tile.  A thread holds at most
    // one 16-column piece of dv (Dv <= 32 kGroups), kept in registers and stored once
    // the next products are issued (plain global stores just before the proxy fence
    // would stall it until they drain)
    uint4 dv_lo = make_uint4(0, 0, 0, 0), dv_hi = dv_lo;
    uint4* dv_dst = nullptr;
    {
      __nv_bfloat16* dvc = (__nv_bfloat16*)p.dv + t0 * p.dv_ld + (int64_t)h * Dv;
      float rs = 0.f;
      acc_walk64(tmp, Dv, len, [&](int s, int col0, float* x) {
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = -x[j];
        __align__(16) __nv_bfloat162 pk[8];
        float vv[16];
        tile_get16(tV, C, s, col0, vv);
#pragma unroll
        for (int j = 0; j < 16; ++j) rs = fmaf(x[j], vv[j], rs);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pk[j] = __floats2bfloat162_rn(bv[s] * x[2 * j], bv[s] * x[2 * j + 1]);
        dv_dst = (uint4*)(dvc + (int64_t)s * p.dv_ld + col0);
        dv_lo = ((const uint4*)pk)[0];
        dv_hi = ((const uint4*)pk)[1];
      });
      rs = x2_pair_sum(rs);
      if (x2_half() == 0) part[grp * C + x2_row()] = rs;
      acc_walk64_8(tmp + 128, C, C, [&](int r, int col0, const float* x) {
        tile_put8(tY, C, r, col0, x);
      });
    }
    __syncthreads();
    if (tid < C) db[tid] += rsum_g(part, tid);
    tc::fence_async_smem();
    mma_issue([&] {
      tc::mma_tile_x(tmp, tc::smem_u32(tT), true, sCC, 64, tc::smem_u32(tdW), true, 8192u, NK, C,
                     0u);                                                         // dBk = T^T dW
      tc::mma_tile_x(tdK, tc::smem_u32(tTW), true, sCC, 64, tc::smem_u32(tdW), true, 8192u, NK,
                     C, 1u);                                                      // dK += b e^G dBk
      tc::mma_tile(tmp + 128, tc::smem_u32(tY), 64, tc::smem_u32(tT), C, C, 0u);  // Y T^T
    }, &bars[0]);
    if (dv_dst != nullptr) {   // this head's dv piece, while the products run
      dv_dst[0] = dv_lo;
      dv_dst[1] = dv_hi;
    }
    ok = mma_wait(&bars[0], mphase, p.status, c);
    if (!ok) break;
    // epilogue D: t_s = rowsum(dBk * K); dA = -(Y T^T) strictly lower.  With
    // A[r][s] = b_r E_rs KK_rs (s < r) and q = dA E KK: db_r += sum_s q[r][s],
    // dG_r += b_r sum_s q[r][s], dG_s -= sum_r b_r q[r][s]; H = dA b_r E for the
    // dK term (H + H^T) K
    {
      float rs = 0.f;
      acc_walk64(tmp, Dk, C, [&](int r, int col0, const float* x) {
        float kv[16];
        tile_get16(tK, C, r, col0, kv);
#pragma unroll
        for (int j = 0; j < 16; ++j) rs = fmaf(kv[j], x[j], rs);
      });
      rs = x2_pair_sum(rs);
      if (x2_half() == 0) part[grp * C + x2_row()] = rs;
      float rq = 0.f;
      acc_walk64_8(tmp + 128, C, C, [&](int r, int s0, const float* x) {
        const float* kkr = sKK + r * KKL + s0;
        float hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s = s0 + j;
          const float E = s < r ? expf(gv[r] - gv[s]) : 0.f;
          const float de = -x[j] * E;            // dA E (zero on and above the diagonal)
          const float qq = de * kkr[j];
          rq += qq;
          X[r * XL + s] = qq * bv[r];
          hv[j] = de * bv[r];
        }
        tile_put8(tH, C, r, s0, hv);
      });
      rq = x2_pair_sum(rq);
      if (x2_half() == 0) rowp[grp * C + x2_row()] = rq;
    }
    __syncthreads();
    {
      const int t = tid & (C - 1), qd = tid / C;
      constexpr int rows = C / kColParts;
      float cs = 0.f;
#pragma unroll 4
      for (int r = qd * rows; r < qd * rows + rows; ++r) cs += X[r * XL + t];
      colp[qd * C + t] = cs;
    }
    __syncthreads();
    if (tid < C) {
      const int t = tid;
      const float ts = rsum_g(part, t), rq = rsum_g(rowp, t);
      float cy = 0.f;
#pragma unroll
      for (int g = 0; g < kColParts; ++g) cy += colp[g * C + t];
      db[t] += ev[t] * ts + rq;
      dG[t] += bv[t] * (ev[t] * ts + rq) - cy;
    }
    tc::fence_async_smem();
    ok = mma_run([&] {
      tc::mma_tile_x(tdK, tc::smem_u32(tH), false, sCC, 64, tc::smem_u32(tK), true, 8192u, NK,
                     C, 1u);                                                      // dK += H K
      tc::mma_tile_x(tdK, tc::smem_u32(tH), true, sCC, 64, tc::smem_u32(tK), true, 8192u, NK,
                     C, 1u);                                                      // dK += H^T K
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // every tile region but K, Q and K K^T is free: the next head's phase A loads run
    // under the gate epilogue
    if (tid == 0 && hh + 1 < p.r) {
      tc::mbar_arrive_expect_tx(&bars[1], phase_a_bytes);
      issue_phase_a_inputs(value_head(p, kh, hh + 1));
      issue_phase_a_walk(value_head(p, kh, hh + 1));
    }
    // gate and sigmoid epilogues: dl = reverse cumsum of dG (one warp, two per lane)
    __syncthreads();
    if (warp == 0) {
      const int l = tid;
      const float a = 2 * l < len ? dG[2 * l] : 0.f, b2 = 2 * l + 1 < len ? dG[2 * l + 1] : 0.f;
      float run = a + b2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, run, o);
        if (l + o < 32) run += y;
      }
      part[2 * l] = run;
      part[2 * l + 1] = run - a;
    }
    __syncthreads();
    {
      float pa = 0.f, pd = 0.f;
      if (tid < len) {
        const int t = tid;
        const float x = xa[t];
        const float ea = expf(al[t]);
        const float l = -ea * softplus_f(x);
        const float dl = part[t];
        const float da = dl * (-ea) * sigmoid_f(x);
        p.dalpha[(t0 + t) * p.dalpha_ld + h] = da;
        p.dbeta[(t0 + t) * p.dbeta_ld + h] = db[t] * bv[t] * (1.f - bv[t]);
        pa = dl * l;
        pd = da;
      }
      pa = warp_sum(pa);
      pd = warp_sum(pd);
      // every read of the scan's sums in part is done past this barrier
      __syncthreads();
      if (tid < C && (tid & 31) == 0) {
        red[tid >> 5] = pa;
        red[2 + (tid >> 5)] = pd;
      }
      __syncthreads();
      if (tid == 0) {
        p.pa[ch] = red[0] + red[1];
        p.pd[ch] = red[2] + red[3];
      }
    }
  }
  // dq, dk of the key head: L2-norm backward of the accumulated dQ_hat, dK_hat,
  // dx = (dx_hat - x_hat (x_hat . dx_hat)) / |x|; the two row dots first, one barrier
  if (ok) {
    {
      float dot[2] = {0.f, 0.f};
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint8_t* xt = which ? tK : tQ;   // x_hat tiles [C][Dk]
        acc_walk64(which ? tdK : tdQ, Dk, C, [&](int r, int col0, const float* x) {
          float xv[16];
          tile_get16(xt, C, r, col0, xv);
#pragma unroll
          for (int j = 0; j < 16; ++j) dot[which] = fmaf(x[j], xv[j], dot[which]);
        });
      }
      dot[0] = x2_pair_sum(dot[0]);
      dot[1] = x2_pair_sum(dot[1]);
      if (x2_half() == 0) {
        part[grp * C + x2_row()] = dot[0];
        rowp[grp * C + x2_row()] = dot[1];
      }
    }
    __syncthreads();
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint8_t* xt = which ? tK : tQ;
      const float* pr = which ? rowp : part;
      __nv_bfloat16* dst = (__nv_bfloat16*)(which ? p.dk : p.dq) +
                           t0 * (which ? p.dk_ld : p.dq_ld) + (int64_t)kh * Dk;
      const int64_t ld = which ? p.dk_ld : p.dq_ld;
      acc_walk64(which ? tdK : tdQ, Dk, len, [&](int r, int col0, const float* x) {
        const float d = rsum_g(pr, r), inv = 1.f / invn[which * C + r];
        __align__(16) __nv_bfloat162 pk[8];
        float xv[16];
        tile_get16(xt, C, r, col0, xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a = (x[2 * j] - xv[2 * j] * d) * inv;
          const float b2 = (x[2 * j + 1] - xv[2 * j + 1] * d) * inv;
          pk[j] = __floats2bfloat162_rn(a, b2);
        }
        uint4* o = (uint4*)(dst + (int64_t)r * ld + col0);
        o[0] = ((const uint4*)pk)[0];
        o[1] = ((const uint4*)pk)[1];
      });
    }
  }
  tc::cp_async_wait_all();   // a unit that stopped early leaves no copy in flight
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_bwd_grads_tc(Params p,
                                                               const __grid_constant__ TmaMaps maps) {
  if (kept_operands_missing(p)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  cta_setup(ctl, 2, 512);
  uint32_t mphase = 0, lphase = 0;
  grads_unit<DK, DV>(p, maps, blockIdx.x, blockIdx.y, base + kCtlBytes, ctl->tmem, ctl->bar, mphase,
                 lphase);
  cta_teardown(ctl, 512);
}

// The backward as one cooperative launch of one CTA per SM, for batches with fewer
// (sequence, value head) walks than SMs: CTAs [0, n_seqs * Hv) walk the chunks in
// reverse and publish each chunk's tiles; the others take (chunk, key head) gradient
// units in descending chunk order from a work counter, each waiting for its chunk's
// flags, and every walk joins them when it is done.  Walks never wait on gradient
// units, so the launch always finishes.
template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_bwd_fused_tc(Params p,
                                                               const __grid_constant__ TmaMaps maps) {
  if (kept_operands_missing(p)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  __shared__ int s_unit;
  cta_setup(ctl, 4, 512);
  const int walks = p.n_seqs * p.Hv;
  if ((int)blockIdx.x < walks) {
    bwd_state_unit<DK, DV>(p, maps, blockIdx.x / p.Hv, blockIdx.x % p.Hv, base + kCtlBytes,
                       ctl->tmem, ctl->bar);
    // fresh mbarriers for the gradient role
    if (threadIdx.x == 0) {
      for (int i = 0; i < 4; ++i) {
        tc::mbar_inval(&ctl->bar[i]);
        tc::mbar_init(&ctl->bar[i], 1);
      }
      tc::fence_mbar_init();
    }
    __syncthreads();
  }
  uint32_t mphase = 0, lphase = 0;
  const int units = p.NC * p.Hk;
  // the next unit is taken while the current one runs
  int next = threadIdx.x == 0 ? (int)atomicAdd(p.bwork, 1u) : 0;
  for (;;) {
    if (threadIdx.x == 0) s_unit = next;
    __syncthreads();
    const int u = s_unit;
    __syncthreads();
    if (u >= units) break;
    if (threadIdx.x == 0) next = (int)atomicAdd(p.bwork, 1u);
    // thread 0 knows the next unit (the others pass a placeholder they do not use)
    const int nc = threadIdx.x == 0 && next < units ? p.NC - 1 - next / p.Hk : -1;
    grads_unit<DK, DV>(p, maps, p.NC - 1 - u / p.Hk, u % p.Hk, base + kCtlBytes, ctl->tmem,
                   ctl->bar, mphase, lphase, nc, threadIdx.x == 0 && next < units ? next % p.Hk : 0);
  }
  cta_teardown(ctl, 512);
}

// d a_log, d dt_bias: one warp per value head; lane l sums chunks l, l + 32, ... in
// order, then a fixed shuffle tree (the same order on every run)
__global__ void k_bwd_gates_tc(Params p) {
  if (kept_operands_missing(p)) return;
  const int lane = threadIdx.x & 31;
  for (int h = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); h < p.Hv;
       h += gridDim.x * (blockDim.x / 32)) {
    float a = 0.f, d = 0.f;
    for (int c = lane; c < p.NC; c += 32) {
      a += p.pa[(size_t)c * p.Hv + h];
      d += p.pd[(size_t)c * p.Hv + h];
    }
    a = warp_sum(a);
    d = warp_sum(d);
    if (lane == 0) {
      p.da_log[h] = a;
      p.ddt_bias[h] = d;
    }
  }
}

// ---------------------------------------------------------------------------
template <int DK>
static size_t bwd_state_tc_smem(const Params& p) {
  const int Dv = p.Dv, MV = Dv < 64 ? 64 : Dv;
  const size_t bK = tc::sw128_bytes(64, DK);
  const size_t bO = (size_t)((Dv + 63) / 64) * 8192;
  const size_t bufsz = bO + 3 * bK + 8192 + 1024;
  return tc::sw128_bytes(MV, DK) + tc::sw128_bytes(64, MV) + 2 * bufsz + 2 * C * 4 + kCtlBytes +
         1024;
}
static size_t grads_tc_smem() {
  return 66560 + 32768 + 49152 + 32768 + 32768 +
         (size_t)((20 + 2 * kGroups + kColParts) * C + kTcThreads / 32) * 4 + kCtlBytes + 1024;
}

template <int DK>
static cudaError_t launch_bwd_state_tc_t(const Params& p, const TmaMaps& maps, cudaStream_t st) {
  const size_t smem = bwd_state_tc_smem<DK>(p);
  auto kern = p.Dv == DK ? k_bwd_state_tc<DK, DK> : k_bwd_state_tc<DK, 0>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_BWD_STATE_TC);
  kern<<<dim3(p.n_seqs, p.Hv), kTcThreads, smem, st>>>(p, maps);
  profile_post(st);
  return cudaGetLastError();
}

// The fused backward (k_bwd_fused_tc) under the same conditions as the fused forward;
// *launched = false otherwise.
template <int DK, int DV>
static cudaError_t launch_bwd_fused_t(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                      bool* launched) {
  *launched = false;
  const int sms = sm_count();
  const int walks = p.n_seqs * p.Hv;
  if (sms <= 0 || walks + kMinProducers > sms || p.NC == 0) return cudaSuccess;
  const size_t a = bwd_state_tc_smem<DK>(p), b = grads_tc_smem();
  const size_t smem = (a > b ? a : b) + 64;
  cudaError_t e = cudaFuncSetAttribute(k_bwd_fused_tc<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_bwd_fused_tc<DK, DV>, kTcThreads, smem);
  if (e != cudaSuccess || per_sm < 1) return cudaSuccess;
  Params pp = p;
  pp.bready = p.bwork + 64;   // the work counter's 256-byte slot, then the flags
  TmaMaps mm = maps;
  void* args[] = {&pp, &mm};
  profile_pre(st, KID_BWD_FUSED_TC);
  e = cudaLaunchCooperativeKernel((const void*)k_bwd_fused_tc<DK, DV>, dim3(sms), dim3(kTcThreads), args,
                                  smem, st);
  profile_post(st);
  if (e == cudaSuccess) *launched = true;
  return e;
}

// The instantiation with the value head size fixed when it equals the key head size.
template <int DK>
static cudaError_t launch_bwd_fused_dk(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                       bool* launched) {
  return p.Dv == DK ? launch_bwd_fused_t<DK, DK>(p, maps, st, launched)
                    : launch_bwd_fused_t<DK, 0>(p, maps, st, launched);
}
template <int DK>
static void (*grads_kernel(const Params& p))(Params, TmaMaps) {
  return p.Dv == DK ? k_bwd_grads_tc<DK, DK> : k_bwd_grads_tc<DK, 0>;
}

cudaError_t launch_bwd_tc(const Params& p, const TmaMaps& maps, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  bool fused = false;
  switch (p.Dk) {
    case 16: e = launch_bwd_fused_dk<16>(p, maps, st, &fused); break;
    case 32: e = launch_bwd_fused_dk<32>(p, maps, st, &fused); break;
    case 64: e = launch_bwd_fused_dk<64>(p, maps, st, &fused); break;
    default: e = launch_bwd_fused_dk<128>(p, maps, st, &fused); break;
  }
  if (e != cudaSuccess) return e;
  if (!fused) {
    if (p.n_seqs > 0) {
      switch (p.Dk) {
        case 16: e = launch_bwd_state_tc_t<16>(p, maps, st); break;
        case 32: e = launch_bwd_state_tc_t<32>(p, maps, st); break;
        case 64: e = launch_bwd_state_tc_t<64>(p, maps, st); break;
        default: e = launch_bwd_state_tc_t<128>(p, maps, st); break;
      }
      if (e != cudaSuccess) return e;
    }
    const size_t smem = grads_tc_smem();
    auto kern = p.Dk == 128 ? grads_kernel<128>(p)
                : p.Dk == 64 ? grads_kernel<64>(p)
                : p.Dk == 32 ? grads_kernel<32>(p)
                             : grads_kernel<16>(p);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    profile_pre(st, KID_BWD_GRADS_TC);
    kern<<<dim3(p.NC, p.Hk), kTcThreads, smem, st>>>(p, maps);
    profile_post(st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  profile_pre(st, KID_BWD_GATES);
  k_bwd_gates_tc<<<(p.Hv + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, st>>>(p);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
