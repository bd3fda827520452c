// gdn_tc_fwd.cu -- tensor-core (tcgen05) forward for bf16 inputs.
//
// k_prep_tc       one CTA per (chunk, key head).  Normalises q, k (L2 with the
//                 1e-6 eps inside the square root), forms [K;Q] K^T on the tensor
//                 core (K K^T and Q K^T in one M = 128 MMA), then for each value
//                 head of the group the gates, T = (I + A)^-1 (blocked forward
//                 substitution in fp32), W^T = K^T diag(b e^G) T^T and
//                 U^T = V^T diag(b) T^T on the tensor core, and P = E * (Q K^T).
//                 Writes bf16 operand tiles (K-major, 128B-swizzled) that the
//                 state walk copies straight into shared memory.
// k_fwd_state_tc  one CTA per (sequence, value head).  Walks the chunks in order
//                 with the state S^T held in registers (fp32) and as a bf16
//                 operand tile; per chunk: X^T = S^T W^T and S^T Q^T (tcgen05),
//                 Delta^T = U^T - X^T, then O^T = diag... P Delta and the state
//                 update S^T <- e^{G_last} S^T + Delta^T diag(c) K (tcgen05).  The
//                 next chunk's tiles are prefetched with the bulk-copy engine
//                 while the current chunk computes.
// Notation as in gdn_internal.cuh; every product is D = A B^T with A, B K-major.
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int C = kChunk;
constexpr int kSeqCache = 1024;   // sequences + 1 whose tables the preparation caches
constexpr int RB = 3;  // value heads prepared together (triangular solves in parallel)

__device__ __forceinline__ size_t tileCD(int D) { return (size_t)((D + 63) / 64) * 64 * 128; }

constexpr int TS = C + 4;   // row stride (floats) of the fp32 [C][C] matrices of the inverse

// In-place inverse T = (I + A)^-1 for nh strictly lower-triangular 64x64 fp32
// matrices A (rows TS floats apart; everything on and above the diagonal zero on
// entry), by 2x2 block inversion at two levels:
//   16x16 diagonal blocks D_b = (I + A_bb)^-1   (forward substitution, a column per thread)
//   32x32 diagonal blocks: lower-left 16x16 = -D_1 A_10 D_0
//   64x64: lower-left 32x32 = -T_B A_BA T_A (T_A, T_B the 32x32 diagonal inverses)
// The 32x32 level runs 1 x 4 register tiles (one row, four columns per thread), the
// 64x64 level 4 x 4 tiles on 2 nh warps.  Scratch M: nh * 1024 floats.  Threads
// 0 .. kTriThreads - 1 call it (all it uses for nh <= RB) and meet on named barrier 1;
// the other warps stay free for work that does not need T.
constexpr int kTriThreads = 128 * RB;
static_assert(kTriThreads % 32 == 0 && kTriThreads < kTcThreads, "warps left beside the inverse");
__device__ void tri_inverse(float* Tm, int nh, float* M) {
  const int tid = threadIdx.x;
  const auto tri_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kTriThreads) : "memory"); };
  // 16x16 diagonal blocks: 16 threads per (head, block), thread j solves column j
  {
    const int unit = tid >> 4, j = tid & 15;
    const bool act = unit < nh * 4;
    float* B = Tm + (act ? (unit >> 2) * C * TS + (unit & 3) * (16 * TS + 16) : 0);
    float x[16];
    if (act) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float a0 = (i == j) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k + 1 < i; k += 2) {
          a0 = fmaf(-B[i * TS + k], x[k], a0);
          a1 = fmaf(-B[i * TS + k + 1], x[k + 1], a1);
        }
        if (i & 1) a0 = fmaf(-B[i * TS + i - 1], x[i - 1], a0);
        x[i] = a0 + a1;
      }
    }
    tri_sync();
    if (act)
#pragma unroll
      for (int i = 0; i < 16; ++i) B[i * TS + j] = x[i];
    tri_sync();
  }
  // 32x32 diagonal blocks (two per head): M = A_10 D_0, then L = -D_1 M.  A thread
  // runs all its 1 x 4 tiles together over the whole k range (the zero triangles
  // add exact zeros), so its accumulators form independent chains.
  {
    constexpr int kMax = (RB * 2 * 16 * 4 + kTcThreads - 1) / kTcThreads;   // tiles per thread
    const int n1 = nh * 2 * 16 * 4;
    float4 acc[kMax];
    int off_a[kMax], off_b[kMax];
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int it = tid + j * kTcThreads;
      const int pr = it < n1 ? it >> 6 : 0, r = (it >> 2) & 15, c0 = (it & 3) * 4;
      const int rb = ((pr & 1) * 2 + 1) * 16, cb = rb - 16;
      off_a[j] = (pr >> 1) * C * TS + (rb + r) * TS + cb;          // row r of A_10
      off_b[j] = (pr >> 1) * C * TS + cb * TS + cb + c0;           // column piece of D_0
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 4
    for (int k = 0; k < 16; ++k)
#pragma unroll
      for (int j = 0; j < kMax; ++j) {
        const float a = Tm[off_a[j] + k];
        const float4 d = *(const float4*)(Tm + off_b[j] + k * TS);
        acc[j].x = fmaf(a, d.x, acc[j].x);
        acc[j].y = fmaf(a, d.y, acc[j].y);
        acc[j].z = fmaf(a, d.z, acc[j].z);
        acc[j].w = fmaf(a, d.w, acc[j].w);
      }
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int it = tid + j * kTcThreads;
      if (it < n1) *(float4*)(M + (it >> 6) * 256 + ((it >> 2) & 15) * 16 + (it & 3) * 4) = acc[j];
    }
    tri_sync();
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int it = tid + j * kTcThreads;
      const int pr = it < n1 ? it >> 6 : 0, r = (it >> 2) & 15;
      const int rb = ((pr & 1) * 2 + 1) * 16;
      off_a[j] = (pr >> 1) * C * TS + (rb + r) * TS + rb;          // row r of D_1
      off_b[j] = pr * 256 + (it & 3) * 4;                          // column piece of M
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 4
    for (int k = 0; k < 16; ++k)
#pragma unroll
      for (int j = 0; j < kMax; ++j) {
        const float d = Tm[off_a[j] + k];
        const float4 m = *(const float4*)(M + off_b[j] + k * 16);
        acc[j].x = fmaf(d, m.x, acc[j].x);
        acc[j].y = fmaf(d, m.y, acc[j].y);
        acc[j].z = fmaf(d, m.z, acc[j].z);
        acc[j].w = fmaf(d, m.w, acc[j].w);
      }
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
      const int it = tid + j * kTcThreads;
      if (it < n1) {
        const int pr = it >> 6, r = (it >> 2) & 15, c0 = (it & 3) * 4;
        const int rb = ((pr & 1) * 2 + 1) * 16, cb = rb - 16;
        *(float4*)(Tm + (pr >> 1) * C * TS + (rb + r) * TS + cb + c0) =
            make_float4(-acc[j].x, -acc[j].y, -acc[j].z, -acc[j].w);
      }
    }
    tri_sync();
  }
  // 64x64: M = A_BA T_A, then lower-left = -T_B M.  Warp w < 2 nh owns a 32 x 16
  // piece of head w / 2 (columns 16 (w % 2) ...); a thread holds the 4 x 4 tile of rows
  // rg + 8i (i < 4) and columns 4 cg ... 4 cg + 3, so a k step costs four broadcast
  // row loads (distinct banks) and one 16-byte column load for 16 FMAs.  T_A is lower
  // triangular: the right half's product starts at k = 16.
  {
    const int w = tid >> 5, l = tid & 31, rg = l >> 2, cg = l & 3;
    const bool act = w < 2 * nh;
    const int hh = act ? w >> 1 : 0, cb = (w & 1) * 16 + cg * 4;
    const float* Th = Tm + hh * C * TS;
    float* Mh = M + hh * 1024;
    float4 acc[4];
    if (act) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int k = (w & 1) * 16; k < 32; ++k) {
        const float4 t = *(const float4*)(Th + k * TS + cb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = Th[(32 + rg + 8 * i) * TS + k];
          acc[i].x = fmaf(a, t.x, acc[i].x);
          acc[i].y = fmaf(a, t.y, acc[i].y);
          acc[i].z = fmaf(a, t.z, acc[i].z);
          acc[i].w = fmaf(a, t.w, acc[i].w);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) *(float4*)(Mh + (rg + 8 * i) * 32 + cb) = acc[i];
    }
    tri_sync();
    if (act) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const float4 m = *(const float4*)(Mh + k * 32 + cb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float t = Th[(32 + rg + 8 * i) * TS + 32 + k];
          acc[i].x = fmaf(t, m.x, acc[i].x);
          acc[i].y = fmaf(t, m.y, acc[i].y);
          acc[i].z = fmaf(t, m.z, acc[i].z);
          acc[i].w = fmaf(t, m.w, acc[i].w);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *(float4*)(Tm + hh * C * TS + (32 + rg + 8 * i) * TS + cb) =
            make_float4(-acc[i].x, -acc[i].y, -acc[i].z, -acc[i].w);
    }
    tri_sync();
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Hand-over between the preparation units one CTA of the fused forward runs in a row,
// as thread 0 sees it.
struct PrepLink {
  int pending;     // the previous unit, whose tile stores may still be in flight and whose
                   // flag is unpublished; -1 if none
  int next;        // the unit this CTA takes next, or -1
  bool kq_issued;  // this unit's raw k / q tiles and its first value head's V tile were
                   // issued by the previous unit
};

// Bytes of prep_unit's buffers (the sequence table follows them).
__host__ __device__ __forceinline__ size_t prep_buffers_bytes(int Dk, int Dv) {
  const size_t b = (size_t)((Dk + 63) / 64) * 128 * 128 + (size_t)((Dv + 63) / 64) * 8192 +
                   2 * 8192;
  return b + sizeof(float) * ((size_t)C * C + (size_t)C * TS + (size_t)RB * C * TS + RB * 1024 +
                              3 * RB * C);
}

// Thread 0: the raw k and q rows of key head kh of the chunk starting at token t0 as TMA
// boxes into the [K; Q] tile, on one phase of `bar`.
__device__ void issue_kq(const Params& p, const TmaMaps& maps, int64_t t0, int kh,
                         uint8_t* tAQK, uint64_t* bar) {
  const int nbk = (p.Dk + 63) / 64;
  tc::mbar_arrive_expect_tx(bar, 2u * nbk * 8192u);
  for (int b = 0; b < nbk; ++b) {
    tc::tma_load_2d(tAQK + b * 128 * 128, &maps.k, kh * p.Dk + 64 * b, (int)t0, bar);
    tc::tma_load_2d(tAQK + b * 128 * 128 + 8192, &maps.q, kh * p.Dk + 64 * b, (int)t0, bar);
  }
}

// Thread 0: the natural V tile of value head j of key head kh (chunk at token t0) into
// `dst`, on one phase of `bar`.
__device__ void issue_v(const Params& p, const TmaMaps& maps, int64_t t0, int kh, int j,
                        uint8_t* dst, uint64_t* bar) {
  const int nbv = (p.Dv + 63) / 64, h = value_head(p, kh, j);
  tc::mbar_arrive_expect_tx(bar, (uint32_t)nbv * 8192u);
  for (int b = 0; b < nbv; ++b)
    tc::tma_load_2d(dst + b * 8192, &maps.v, h * p.Dv + 64 * b, (int)t0, bar);
}

// One (chunk c, key head kh) unit of the preparation on a whole CTA.  `sm` is its
// shared memory (1024-aligned, prep_tc_smem bytes, ending in the sequence table `tab`
// may point to), `tmem` 256 TMEM columns, bar[0] /
// bar[1] the MMA and k / q load mbarriers with their running phases, bar[2] / bar[3] the
// two V buffers' (phases in bits 0 / 1 of vphase).  The value heads' V tiles land ahead
// of use: head 0's with the k / q rows, the next head's in the second buffer (the K K^T
// region, free once A is formed; only when the unit's heads form one group) and the
// head after that as soon as the product of the head before it has read the buffer.
// Every workspace tile leaves by plain stores from the threads that form it (the
// natural K / Q tiles at the normalisation, K K^T at the Gram epilogue, diag(c) K, P and
// the backward's T tiles while a head's products run, W and U^T at its epilogue): no
// bulk store, so the copy engine serves the loads alone.  Without `link` the unit's
// writes are done when the kernel ends.  With it (fused forward) the unit publishes
// link->pending's flag (that unit's writes all came before this unit's CTA barriers)
// once the inverse's inputs are formed, and issues link->next's k / q tiles and first V
// tile once its last product has read its own (setting link->kq_issued; link->next is
// the raw work-counter value, a unit index only below NC Hk).  False after a timed-out
// wait.
template <int DK, int DV>   // DV: the value head size when fixed, else 0 (p.Dv)
__device__ bool prep_unit(const Params& p, const TmaMaps& maps, const SeqTab& tab, int bwd,
                          int c, int kh, uint8_t* sm, uint32_t tmem, uint64_t* bar,
                          uint32_t& phase, uint32_t& lphase, uint32_t& vphase, PrepLink* link) {
  int n;
  int64_t t0;
  int len;
  __shared__ int s_publish;   // the previous unit, handed from thread 0 to its publisher
  const bool kq_issued = link != nullptr && link->kq_issued;
  if (link != nullptr && threadIdx.x == 0) link->kq_issued = false;
  if (!chunk_info(p, tab, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return true;
  }
  constexpr int Dk = DK;   // the head sizes p.Dk, p.Dv, fixed by the instantiation where it can
  const int Dv = DV > 0 ? DV : p.Dv;
  const int MV = Dv < 64 ? 64 : Dv;
  constexpr int NK = Dk < 64 ? 64 : Dk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nbk = (Dk + 63) / 64, nbv = (Dv + 63) / 64;
  const uint32_t aqk_pitch = 128u * 128u;               // 64-column blocks of the [K; Q] tile
  const uint32_t bKC = tc::sw128_bytes(64, Dk);
  uint8_t* tAQK = sm;                                   // [128][Dk]: rows 0-63 K, 64-127 Q
  uint8_t* sV = tAQK + nbk * aqk_pitch;                 // [C][Dv] natural V of one head (TMA)
  uint8_t* tTW = sV + nbv * 8192;                       // [C][C] T diag(b e^G)
  uint8_t* tTB = tTW + 8192;                            // [C][C] T diag(b)
  float* KK = (float*)(tTB + 8192);                     // [C][C]
  float* QK = KK + C * C;                               // [C][TS]
  float* Tm = QK + C * TS;                              // [RB][C][TS]
  float* Mt = Tm + RB * C * TS;                         // [RB][1024] scratch of the inverse
  float* gv = Mt + RB * 1024;                           // [RB][C]
  float* bv = gv + RB * C;                              // [RB][C]
  float* wv = bv + RB * C;                              // [RB][C]

  __syncthreads();
  // TMEM columns: [0, 64) the Gram products, [64, 64 + NK) W, [192, 256) U^T
  const uint32_t tAccW = tmem + 64, tAccU = tmem + 192;
  bool ok = true;
  // the first head group's raw gate inputs, loaded while the q/k tiles are in flight
  float pre_beta = 0.f, pre_x = 0.f, pre_al = 0.f;
  {
    const int nh0 = p.r < RB ? p.r : RB;
    if (tid < nh0 * C && tid % C < len) {
      const int t = tid % C, h = value_head(p, kh, tid / C);
      pre_beta = p.beta_raw[(t0 + t) * p.beta_ld + h];
      pre_x = p.alpha[(t0 + t) * p.alpha_ld + h] + p.dt_bias[h];
      pre_al = p.a_log[h];
    }
  }
  const size_t ckk = (size_t)c * p.Hk + kh, ck = ckk * C;
  // raw k and q rows of the chunk: TMA boxes straight into the [K; Q] operand tile
  // (issued by the previous unit when it could)
  if (tid == 0 && !kq_issued) {
    issue_kq(p, maps, t0, kh, tAQK, &bar[1]);
    issue_v(p, maps, t0, kh, 0, sV, &bar[2]);
  }
  // the unit's value heads form one group of at most RB: odd heads take the second buffer
  const bool two_v = p.r <= RB;
  {
    const bool lok = tc::mbar_wait(&bar[1], lphase);
    lphase ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
      ok = false;
    }
  }
  if (!ok) goto done;

  // 1. L2 normalisation in place, four threads per row (K rows 0-63, Q rows 64-127),
  // each with its share of the row's 16-byte pieces in registers; rows past the
  // chunk become zero
  {
    const int row = tid >> 2, part = tid & 3;
    const int nch = Dk / 8, tpr = nch < 4 ? nch : 4, cpt = part < tpr ? nch / tpr : 0;
    const bool isq = row >= C;
    const int t = row & (C - 1);
    uint4 raw[4];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < cpt) {
        raw[j] = *(const uint4*)(tAQK + tc::sw128_offset(row, (part * cpt + j) * 8, 128));
        const __nv_bfloat162* e = (const __nv_bfloat162*)&raw[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(e[q]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float nrm = sqrtf(ss + 1e-6f), inv = t < len ? 1.f / nrm : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < cpt) {
        const __nv_bfloat162* e = (const __nv_bfloat162*)&raw[j];
        __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(e[q]);
          pk[q] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
        }
        *(uint4*)(tAQK + tc::sw128_offset(row, (part * cpt + j) * 8, 128)) = *(const uint4*)pk;
      }
    if (bwd && part == 0) (isq ? p.nq : p.nk)[ck + t] = nrm;
    // Dk < 64: the box's columns past Dk (a neighbouring head) become zero padding
    if (Dk < 64) {
      const int padc = 8 - Dk / 8;
      for (int idx = tid; idx < 2 * C * padc; idx += kTcThreads) {
        const int row = idx / padc, c0 = (Dk / 8 + idx % padc) * 8;
        *(uint4*)(tAQK + tc::sw128_offset(row, c0, 128)) = make_uint4(0, 0, 0, 0);
        *(uint4*)((row >= C ? p.Qsw : p.Ksw) + ckk * bKC + tc::sw128_offset(row & (C - 1), c0, 64)) =
            make_uint4(0, 0, 0, 0);
      }
    }
  }
  tc::fence_async_smem();
  __syncthreads();
  // 2. [K; Q] K^T -> TMEM columns [0, 64): lanes 0-63 K K^T, lanes 64-127 Q K^T.
  mma_issue([&] { tc::mma_tile_p(tmem, tc::smem_u32(tAQK), aqk_pitch, 128, tc::smem_u32(tAQK),
                                 aqk_pitch, 64, Dk, 0u); },
            &bar[0]);
  {
    // the natural K and Q tiles of the key head into the workspace while the product
    // runs (plain stores issued before the proxy fence above would have stalled it):
    // each thread copies the pieces it normalised
    const int row = tid >> 2, part = tid & 3;
    const int nch = Dk / 8, tpr = nch < 4 ? nch : 4, cpt = part < tpr ? nch / tpr : 0;
    uint8_t* dst = (row >= C ? p.Qsw : p.Ksw) + ckk * bKC;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < cpt) {
        const int k8 = (part * cpt + j) * 8;
        *(uint4*)(dst + tc::sw128_offset(row & (C - 1), k8, 64)) =
            *(const uint4*)(tAQK + tc::sw128_offset(row, k8, 128));
      }
  }
  ok = mma_wait(&bar[0], phase, p.status, c);
  if (!ok) goto done;
  acc_walk(tmem, 128, 64, 128, [&](int row, int col0, const float* v) {
    float* dst = row < C ? KK + row * C : QK + (row - C) * TS;
    *(float4*)(dst + col0) = make_float4(v[0], v[1], v[2], v[3]);
    *(float4*)(dst + col0 + 4) = make_float4(v[4], v[5], v[6], v[7]);
    *(float4*)(dst + col0 + 8) = make_float4(v[8], v[9], v[10], v[11]);
    *(float4*)(dst + col0 + 12) = make_float4(v[12], v[13], v[14], v[15]);
    if (bwd && row < C) {   // K K^T (fp32, row-major) for the gradient kernel
      float* g = p.KKf + (ck + row) * C + col0;
      *(float4*)(g) = make_float4(v[0], v[1], v[2], v[3]);
      *(float4*)(g + 4) = make_float4(v[4], v[5], v[6], v[7]);
      *(float4*)(g + 8) = make_float4(v[8], v[9], v[10], v[11]);
      *(float4*)(g + 12) = make_float4(v[12], v[13], v[14], v[15]);
    }
  });
  __syncthreads();

  for (int g0 = 0; g0 < p.r; g0 += RB) {
    const int nh = (p.r - g0) < RB ? (p.r - g0) : RB;
    // 3. gates of the nh value heads
    if (tid < nh * C) {
      const int hh = tid / C, t = tid % C, h = value_head(p, kh, g0 + hh);
      float l = 0.f, b = 0.f;
      if (t < len) {
        const float braw = g0 == 0 ? pre_beta : p.beta_raw[(t0 + t) * p.beta_ld + h];
        const float x = g0 == 0 ? pre_x : p.alpha[(t0 + t) * p.alpha_ld + h] + p.dt_bias[h];
        b = sigmoid_f(braw);
        l = -expf(g0 == 0 ? pre_al : p.a_log[h]) * softplus_f(x);
      }
      gv[hh * C + t] = l;
      bv[hh * C + t] = b;
    }
    __syncthreads();
    if (warp < nh && lane < 32) {
      // inclusive cumsum of 64 values, two per lane
      float* x = gv + warp * C;
      const float a = x[2 * lane], b2 = a + x[2 * lane + 1];
      float run = b2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, run, o);
        if (lane >= o) run += y;
      }
      x[2 * lane] = run - b2 + a;
      x[2 * lane + 1] = run;
    }
    __syncthreads();
    if (tid < nh * C) {
      const int hh = tid / C, t = tid % C, h = value_head(p, kh, g0 + hh);
      const size_t ch = (size_t)c * p.Hv + h;
      wv[hh * C + t] = bv[hh * C + t] * expf(gv[hh * C + t]);
      p.G[ch * C + t] = gv[hh * C + t];
      p.b[ch * C + t] = bv[hh * C + t];
    }
    // A = diag(b) (E * K K^T), strictly lower, four columns per step (C * C / 4 pieces a
    // head: two passes of the CTA)
    static_assert(C * C / 4 == 2 * kTcThreads, "two passes a head");
#pragma unroll 2
    for (int it = 0; it < 2 * nh; ++it) {
      const int idx = tid + it * kTcThreads;
      const int hh = idx / (C * C / 4), e4 = idx % (C * C / 4), r = e4 / (C / 4), s0 = (e4 % (C / 4)) * 4;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 < r) {
        const float* g = gv + hh * C;
        const float br = bv[hh * C + r], gr = g[r];
        const float4 kk = *(const float4*)(KK + r * C + s0);
        const float4 gs = *(const float4*)(g + s0);
        // the exponent is at most 0: the intrinsic's error (a few ulp) is far below the
        // bf16 rounding every product operand takes later
        a.x = br * __expf(gr - gs.x) * kk.x;
        if (s0 + 1 < r) a.y = br * __expf(gr - gs.y) * kk.y;
        if (s0 + 2 < r) a.z = br * __expf(gr - gs.z) * kk.z;
        if (s0 + 3 < r) a.w = br * __expf(gr - gs.w) * kk.w;
      }
      *(float4*)(Tm + hh * C * TS + r * TS + s0) = a;
    }
    // the previous unit goes for its publication to the inverse's last thread, which its
    // first (16x16) phase leaves idle, so that the fence holds up no one
    if (g0 == 0 && tid == 0) {
      s_publish = link != nullptr ? link->pending : -1;
      if (link != nullptr) link->pending = -1;
    }
    tc::fence_async_smem();   // the K K^T reads come before the V tile that replaces it
    __syncthreads();
    static_assert(kTriThreads - 1 >= 64 * RB, "the publisher sits out the 16x16 phase");
    if (g0 == 0 && tid == kTriThreads - 1) {
      // every write of the previous unit came before this CTA's barriers: publish it
      if (s_publish >= 0) publish_flag(p.fready + s_publish);
      if (two_v && p.r > 1) issue_v(p, maps, t0, kh, 1, (uint8_t*)KK, &bar[3]);
    }
    // 4. T = (I + A)^-1 for the nh heads at once, while warps 12-15 write every head's
    // diag(c) K with c_s = e^{G_last - G_s} (zero past the chunk), the operand the walk's
    // state update S <- e^{G_last} S + (diag(c) K)^T Delta takes
    if (tid < kTriThreads) {
      tri_inverse(Tm, nh, Mt);
    } else {
      constexpr int nt = kTcThreads - kTriThreads;
      const int t3 = tid - kTriThreads, c8n = NK / 8;
      for (int hh = 0; hh < nh; ++hh) {
        const float* G = gv + hh * C;
        const float gl = G[len - 1];
        uint8_t* dst = p.Kcw + ((size_t)c * p.Hv + value_head(p, kh, g0 + hh)) * bKC;
        for (int idx = t3; idx < C * c8n; idx += nt) {
          const int s = idx / c8n, k8 = (idx % c8n) * 8;
          const uint4 raw = *(const uint4*)(tAQK + tc::sw128_offset(s, k8, 128));
          const __nv_bfloat162* e = (const __nv_bfloat162*)&raw;
          const float cs = s < len ? __expf(gl - G[s]) : 0.f;
          __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(e[q]);
            pk[q] = __floats2bfloat162_rn(f.x * cs, f.y * cs);
          }
          *(uint4*)(dst + tc::sw128_offset(s, k8, C)) = *(const uint4*)pk;
        }
      }
    }
    __syncthreads();
    // 5. per head: W = T diag(w) K, U^T = V^T (T diag(b))^T, P
    for (int hh = 0; hh < nh; ++hh) {
      const int h = value_head(p, kh, g0 + hh);
      const size_t ch = (size_t)c * p.Hv + h;
      const float* T = Tm + hh * C * TS;
      const int j = g0 + hh;
      const bool odd = two_v && (j & 1);
      uint8_t* vb = odd ? (uint8_t*)KK : sV;   // this head's V tile
      if (tid == 0) {
        // the maps of the loads this head issues after its products
        tc::prefetch_tensormap(&maps.v);
        if (j + 1 == p.r) {
          tc::prefetch_tensormap(&maps.k);
          tc::prefetch_tensormap(&maps.q);
        }
      }
      __syncthreads();
      const float* w = wv + hh * C;
      const float* bb = bv + hh * C;
      const float* G = gv + hh * C;
      // T diag(w) and T diag(b) into the product tiles; P, and for the backward T and
      // T diag(w), stay in registers and go to the workspace while the products run.
      // Thread tid takes row r = tid / 8, columns [s8, s8 + 8) with s8 = 8 (tid % 8), so
      // eight threads fill a row of each tile (one 128-byte line of the workspace copy).
      static_assert(C * C / 8 == kTcThreads, "one 8-column piece of the C x C tiles a thread");
      uint4 rp, rt, rw;
      uint32_t toff;
      {
        const int r = tid >> 3, s8 = (tid & 7) * 8;
        const float4 ta = *(const float4*)(T + r * TS + s8);
        const float4 tb = *(const float4*)(T + r * TS + s8 + 4);
        const float4 qa = *(const float4*)(QK + r * TS + s8);
        const float4 qb = *(const float4*)(QK + r * TS + s8 + 4);
        const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const float gr = G[r];
        __align__(16) __nv_bfloat162 pw[4], pb[4], pp[4], pt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s = s8 + 2 * u;
          pw[u] = __floats2bfloat162_rn(tv[2 * u] * w[s], tv[2 * u + 1] * w[s + 1]);
          pb[u] = __floats2bfloat162_rn(tv[2 * u] * bb[s], tv[2 * u + 1] * bb[s + 1]);
          pp[u] = __floats2bfloat162_rn(s <= r ? __expf(gr - G[s]) * qv[2 * u] : 0.f,
                                        s + 1 <= r ? __expf(gr - G[s + 1]) * qv[2 * u + 1] : 0.f);
          pt[u] = __floats2bfloat162_rn(tv[2 * u], tv[2 * u + 1]);
        }
        toff = tc::sw128_offset(r, s8, C);
        *(uint4*)(tTW + toff) = *(const uint4*)pw;
        *(uint4*)(tTB + toff) = *(const uint4*)pb;
        rp = *(const uint4*)pp;
        rt = *(const uint4*)pt;
        rw = *(const uint4*)pw;
      }
      {
        const uint32_t bit = odd ? 2u : 1u;
        const bool lok = tc::mbar_wait(odd ? &bar[3] : &bar[2], (vphase & bit) ? 1u : 0u);
        vphase ^= bit;
        if (__syncthreads_or(lok ? 0 : 1)) {
          if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
          ok = false;
          goto done;
        }
      }
      // rows of the V tile past the chunk (another sequence's tokens) read as zero
      if (len < C)
        for (int idx = tid; idx < nbv * (C - len) * 8; idx += kTcThreads) {
          const int b2 = idx / ((C - len) * 8), rem = idx % ((C - len) * 8);
          ((uint4*)(vb + b2 * 8192 + (len + rem / 8) * 128))[rem % 8] = make_uint4(0, 0, 0, 0);
        }
      tc::fence_async_smem();
      mma_issue([&] {
        // W = (T diag(w)) K: B is K read MN-major from the rows of the [K; Q] tile
        tc::mma_tile_x(tAccW, tc::smem_u32(tTW), false, 8192u, 64, tc::smem_u32(tAQK), true,
                       aqk_pitch, NK, C, 0u);
        // U^T = V^T (T diag(b))^T: A is V^T read MN-major from the natural V tile
        tc::mma_tile_x(tAccU, tc::smem_u32(vb), true, 8192u, MV, tc::smem_u32(tTB), false,
                       8192u, C, C, 0u);
      }, &bar[0]);
      // the tiles that only the workspace takes leave while the products run (after the
      // proxy fence above, which therefore never waits for them)
      *(uint4*)(p.Psw + ch * 8192 + toff) = rp;
      if (bwd) {
        *(uint4*)(p.Tb + ch * 16384 + toff) = rt;
        *(uint4*)(p.Tb + ch * 16384 + 8192 + toff) = rw;
      }
      ok = mma_wait(&bar[0], phase, p.status, c);
      if (!ok) goto done;
      if (tid == 0) {
        // this head's V buffer is free again: the next head that uses it may land
        const int jn = two_v ? j + 2 : j + 1;
        if (!odd && jn < p.r) issue_v(p, maps, t0, kh, jn, sV, &bar[2]);
        // the unit's last product has read the [K; Q] tile and the V tiles: the next
        // unit's rows and first V tile may land
        if (link != nullptr && j + 1 == p.r && link->next >= 0 && link->next < p.NC * p.Hk) {
          const int cn = link->next / p.Hk, khn = link->next % p.Hk;
          int nn, nlen;
          int64_t nt0;
          if (chunk_info(p, tab, cn, &nn, &nt0, &nlen)) {
            issue_kq(p, maps, nt0, khn, tAQK, &bar[1]);
            issue_v(p, maps, nt0, khn, 0, sV, &bar[2]);
            link->kq_issued = true;
          }
        }
      }
      acc_walk64(tAccW, Dk, C, [&](int s, int col0, const float* v) {
        tile_put16(p.Wsw + ch * bKC, C, s, col0, v);
      });
      if (Dk < 64)   // the W tile's padding columns
        for (int idx = tid; idx < C * (8 - Dk / 8); idx += kTcThreads) {
          const int s = idx / (8 - Dk / 8), c0 = (Dk / 8 + idx % (8 - Dk / 8)) * 8;
          *(uint4*)(p.Wsw + ch * bKC + tc::sw128_offset(s, c0, C)) = make_uint4(0, 0, 0, 0);
        }
      acc_walk(tAccU, MV, 64, Dv, [&](int vv, int col0, const float* v) {
        // U^T as a [Dv][C] SW128 tile, so that row reads by the state walks are conflict-free
        tile_put16((uint8_t*)(p.Utb + ch * Dv * C), Dv, vv, col0, v);
      });
    }
  }
done:
  if (tid == 0 && link == nullptr) tc::bulk_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  return ok;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_prep_tc(Params p,
                                                          const __grid_constant__ TmaMaps maps,
                                                          int bwd) {
  stamp_kept_operands(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  cta_setup(ctl, 4, 256);
  uint32_t phase = 0, lphase = 0, vphase = 0;
  const SeqTab tab =
      seq_tab(p, (int32_t*)(base + kCtlBytes + prep_buffers_bytes(p.Dk, p.Dv)), kSeqCache);
  prep_unit<DK, DV>(p, maps, tab, bwd, blockIdx.x, blockIdx.y, base + kCtlBytes, ctl->tmem,
                ctl->bar, phase, lphase, vphase, nullptr);
  cta_teardown(ctl, 256);
}

// ---------------------------------------------------------------------------
// The chunk walk of sequence n, value head h on a whole CTA (`sm`: 1024-aligned,
// fwd_state_tc_smem bytes; `tmem`: 512 columns; bars[0..2]: MMA and the two load
// buffers).  In a fused launch (p.fready set) chunk c's tiles are read only after the
// preparation unit (c, key head) has published them.  The walk carries only the state:
// per chunk it writes the chunk-start state (fp32, and as a bf16 S^T tile) and the
// Delta^T tile, from which the output pass (out_unit) forms O.  Every one of these
// leaves by a bulk store from shared memory (the fp32 state through two staging
// buffers): global stores issued by the threads themselves would hold up their next
// proxy fence until they drain.
template <int DK, int DV>   // DV: the value head size when fixed, else 0 (p.Dv)
__device__ void fwd_state_unit(const Params& p, int n, int h, uint8_t* sm, uint32_t tmem,
                               uint64_t* bars) {
  const int kh = key_head(p, h);
  int64_t s0, s1;
  int c0, c1;
  if (!seq_info(p, n, &s0, &s1, &c0, &c1)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, n);
    return;
  }
  constexpr int NKC = (DK + 16 * kGroups - 1) / (16 * kGroups);   // S^T pieces per thread
  constexpr int NKF = DK < 64 ? 64 : DK;        // N of products read K MN-major
  const int Dv = DV > 0 ? DV : p.Dv, MV = Dv < 64 ? 64 : Dv;
  const int tid = threadIdx.x, grp = col_group();
  const uint32_t bW = (uint32_t)tileCD(DK);
  // G slot: the chunk's G (C floats), or e^{G_last} per channel for KDA (DK floats)
  constexpr int EVS = DK > C ? DK : C;
  const uint32_t bU = (uint32_t)Dv * C * 2, bG = EVS * 4, gbytes = (p.kda ? DK : C) * 4;
  const uint32_t bSt = tc::sw128_bytes(MV, DK);       // one saved S^T tile
  uint8_t* tSt = sm;                                  // [MV][DK]
  uint8_t* buf0 = tSt + tc::sw128_bytes(MV, DK);
  const uint32_t bufsz = bW * 2 + ((bU + bG + 1023) & ~1023u);
  uint8_t* tDt = buf0 + 2 * bufsz;                    // [MV][C] Delta^T
  const uint32_t bHalf = (uint32_t)(DK / 2) * Dv * 4; // half an fp32 state
  float* stg0 = (float*)(tDt + MV * 128);             // [DK / 2][Dv] fp32 staging, rows
  float* stg1 = (float*)((uint8_t*)stg0 + ((bHalf + 1023) & ~1023u));   // 0.. and DK/2..
  float* evb = (float*)((uint8_t*)stg1 + ((bHalf + 1023) & ~1023u));   // [2][EVS] decay
  auto tW = [&](int b) { return buf0 + b * bufsz; };
  auto tK = [&](int b) { return buf0 + b * bufsz + bW; };   // diag(c) K of the value head
  auto sU = [&](int b) { return (const __nv_bfloat16*)(buf0 + b * bufsz + 2 * bW); };
  auto sG = [&](int b) { return (const float*)(buf0 + b * bufsz + 2 * bW + bU); };
  const uint32_t bDt = (uint32_t)MV * 128;            // one Delta^T tile

  for (int i = tid; i < (int)(tc::sw128_bytes(MV, DK) / 16); i += kTcThreads)
    ((uint4*)tSt)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < MV * 128 * 2 / 16; i += kTcThreads) ((uint4*)tDt)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // TMEM: X = S^T W^T @0, state update @64
  const uint32_t tX = tmem, tS = tmem + 64;
  uint32_t mphase = 0, lph[2] = {0, 0};
  const bool f32_states = p.saved && !p.bf16_states;
  const int vrow = acc_row(MV);
  const bool vok = vrow >= 0 && vrow < Dv;
  const size_t SZ = (size_t)DK * Dv;

  // state S^T (row v = this thread's lane, columns k of its 16-column pieces)
  float S[NKC][16];
#pragma unroll
  for (int i = 0; i < NKC; ++i)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int k = grp * 16 + 16 * kGroups * i + j;
      S[i][j] = (vok && k < DK && p.S0) ? p.S0[((size_t)n * p.Hv + h) * SZ + (size_t)k * Dv + vrow] : 0.f;
    }
#pragma unroll
  for (int i = 0; i < NKC; ++i)
    if (grp * 16 + 16 * kGroups * i < DK && vok)
      tile_put16(tSt, MV, vrow, grp * 16 + 16 * kGroups * i, S[i]);
  tc::fence_async_smem();

  auto issue_load = [&](int cc, int b) {
    uint64_t* lb = &bars[1 + b];
    const size_t chh = (size_t)cc * p.Hv + h;
    tc::mbar_arrive_expect_tx(lb, 2 * bW + bU + gbytes);
    tc::bulk_g2s(tW(b), p.Wsw + chh * bW, bW, lb);
    tc::bulk_g2s(tK(b), p.Kcw + chh * bW, bW, lb);
    tc::bulk_g2s((void*)sU(b), p.Utb + chh * Dv * C, bU, lb);
    if (p.kda)
      tc::bulk_g2s((void*)sG(b), p.Gl + chh * DK, gbytes, lb);
    else
      tc::bulk_g2s((void*)sG(b), p.G + chh * C, gbytes, lb);
  };
  // Thread 0 issues chunk loads in order; a fused launch first needs the preparation
  // unit's flag (blocking only when the walk cannot go on without the chunk).
  int issued = c0 - 1, acquired = c0 - 1;   // acquired: the flag was already read set
  int opub = c0;   // thread 0: chunks [c0, opub) are published for the output units
  auto try_issue = [&](int cc, bool block) {
    if (cc >= c1 || cc != issued + 1) return;
    if (p.fready && cc == acquired) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
    } else if (p.fready) {
      const uint32_t* f = p.fready + (size_t)cc * p.Hk + kh;
      if (block) {
        if (!wait_flag(f)) set_status(p.status, GDN_ERR_TIMEOUT, cc);
      } else if (!flag_ready(f)) {
        return;
      } else {
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
    }
    issue_load(cc, (cc - c0) & 1);
    issued = cc;
  };
  auto chunk_len = [&](int cc) {
    const int64_t t = s0 + (int64_t)(cc - c0) * C;
    return (int)((s1 - t) < C ? (s1 - t) : C);
  };
  // Brings chunk cc's tiles in (waits for them), fills its gate vectors, stores its
  // chunk-start state and issues its first product X = S^T W^T.  Returns false on a
  // timed-out wait.
  auto start_chunk = [&](int cc) -> bool {
    const int b = (cc - c0) & 1, len = chunk_len(cc);
    if (tid == 0) try_issue(cc, true);
    const bool lok = tc::mbar_wait(&bars[1 + b], lph[b]);
    lph[b] ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, cc);
      return false;
    }
    const float* G = sG(b);
    // the state's decay over the chunk: e^{G_last} (or, for KDA, per channel)
    if (p.kda) {
      if (tid < DK) evb[b * EVS + tid] = G[tid];
    } else if (tid == 0) {
      evb[b * EVS] = expf(G[len - 1]);
    }
    mma_issue([&] {
      // the previous chunk's Delta^T store has read its tile (the epilogue after this
      // product rewrites it); its two fp32 halves, stored after it, may still be read
      if (f32_states) tc::bulk_wait_read<2>();
      else tc::bulk_wait_read<0>();
      tc::mma_tile(tX, tc::smem_u32(tSt), MV, tc::smem_u32(tW(b)), C, DK, 0u);
      // the chunk-start state as a bf16 S^T tile, for the output pass and the backward:
      // the saved state itself (GDN_FLAG_BF16_SAVED_STATES) or the workspace copy; one
      // bulk store issued behind the product (the two would contend for the tile's reads)
      uint8_t* tile_dst = p.saved && p.bf16_states ? (uint8_t*)p.saved : p.Stb;
      tc::bulk_s2g(tile_dst + ((size_t)cc * p.Hv + h) * bSt, tSt, bSt);
      tc::bulk_commit();
    }, &bars[0]);
    return true;
  };

  bool ok = true;
  if (c1 > c0) {
    if (tid == 0) {
      try_issue(c0, true);
      try_issue(c0 + 1, false);
    }
    ok = start_chunk(c0);
  }
  // Half `half` (rows k of S in [half DK/2, half DK/2 + DK/2)) of the fp32 state in the
  // registers into its staging buffer [DK/2][Dv] (a warp's lanes write consecutive v)
  auto stage_halves = [&]() {
    if (!vok) return;
#pragma unroll
    for (int ii = 0; ii < NKC; ++ii) {
      const int k0 = grp * 16 + 16 * kGroups * ii;
      if (k0 < DK)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int k = k0 + j;
          float* dst = k < DK / 2 ? stg0 + (size_t)k * Dv : stg1 + (size_t)(k - DK / 2) * Dv;
          dst[vrow] = S[ii][j];
        }
    }
  };
  for (int c = c0; c < c1 && ok; ++c) {
    const int i = c - c0, b = i & 1;
    const int len = chunk_len(c);
    // the staging buffers' last stores have read them (the barrier below orders this
    // before the next writes); the state tile's store may still be reading
    if (tid == 0 && f32_states) tc::bulk_wait_read<1>();
    // fused launch, every eighth chunk: the groups older than the last chunk's (its
    // Delta^T tile and fp32 halves) and this chunk's state tile have landed, so chunks
    // up to c - 2 are complete for the output units: one fence for the run
    if (tid == 0 && p.oready && i > 1 && (i & 7) == 0) {
      if (f32_states)
        tc::bulk_wait<4>();
      else
        tc::bulk_wait<2>();
      publish_flags(p.oready + (size_t)opub * p.Hv + h, (size_t)p.Hv, c - 1 - opub);
      opub = c - 1;
    }
    ok = mma_wait(&bars[0], mphase, p.status, c);
    if (!ok) break;
    // Delta^T = U^T - X^T
    const uint8_t* U = (const uint8_t*)sU(b);
#pragma unroll
    for (int q = 0; q < C / (16 * kGroups); ++q) {
      const int col0 = grp * 16 + 16 * kGroups * q;
      float x[16];
      tc::tmem_ld16(tX + lane_quarter() + col0, x);
      tc::tmem_ld_wait();
      if (vok) {
        float u[16];
        tile_get16(U, Dv, vrow, col0, u);
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = u[j] - x[j];
        tile_put16(tDt, MV, vrow, col0, x);
      }
    }
    // the chunk's fp32 start state, still in the registers, into the staging buffers
    if (f32_states) stage_halves();
    tc::fence_async_smem();
    // the state update; the Delta^T tile and the fp32 state go out
    ok = mma_run([&] {
      tc::bulk_wait_read<0>();   // the state tile's store has read S^T: the update may rewrite it
      // (diag(c) K)^T read MN-major from the natural tile
      tc::mma_tile_x(tS, tc::smem_u32(tDt), false, (uint32_t)MV * 128u, MV, tc::smem_u32(tK(b)),
                     true, 8192u, NKF, C, 0u);
      tc::bulk_s2g(p.Dtb + ((size_t)c * p.Hv + h) * bDt, tDt, bDt);
      tc::bulk_commit();
      if (f32_states) {
        float* dst = p.saved + ((size_t)c * p.Hv + h) * SZ;
        tc::bulk_s2g(dst, stg0, bHalf);
        tc::bulk_commit();
        tc::bulk_s2g(dst + (size_t)(DK / 2) * Dv, stg1, bHalf);
        tc::bulk_commit();
      }
      // while the tensor core works: is chunk c + 2 prepared (flag read ahead)?
      if (p.fready && c + 2 < c1 && issued == c + 1 &&
          flag_ready(p.fready + (size_t)(c + 2) * p.Hk + kh))
        acquired = c + 2;
    }, &bars[0], mphase, p.status, c);
    if (!ok) break;
    // buffer b is free (no tile of chunk c is read from here on): chunk c + 2's tiles
    if (tid == 0) {
      try_issue(c + 1, false);
      try_issue(c + 2, false);
    }
    // S^T <- e^{G_last} S^T + Delta^T diag(c) K
    const float eC = evb[b * EVS];
#pragma unroll
    for (int ii = 0; ii < NKC; ++ii) {
      const int col0 = grp * 16 + 16 * kGroups * ii;
      if (col0 < DK) {
        float x[16];
        tc::tmem_ld16(tS + lane_quarter() + col0, x);
        tc::tmem_ld_wait();
        if (vok) {
          if (p.kda) {   // row k of S decays by its own channel's gate
#pragma unroll
            for (int j = 0; j < 16; ++j) S[ii][j] = fmaf(evb[b * EVS + col0 + j], S[ii][j], x[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) S[ii][j] = fmaf(eC, S[ii][j], x[j]);
          }
          tile_put16(tSt, MV, vrow, col0, S[ii]);
        }
      }
    }
    tc::fence_async_smem();
    if (c + 1 < c1 && !start_chunk(c + 1)) {
      ok = false;
      break;
    }
  }
  if (ok && p.S_T && vok)
#pragma unroll
    for (int ii = 0; ii < NKC; ++ii)
      if (grp * 16 + 16 * kGroups * ii < DK)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          p.S_T[((size_t)n * p.Hv + h) * SZ + (size_t)(grp * 16 + 16 * kGroups * ii + j) * Dv +
                vrow] = S[ii][j];
  if (tid == 0) {
    tc::bulk_wait<0>();
    // the rest (also after an error: the status word then holds it)
    if (p.oready) publish_flags(p.oready + (size_t)opub * p.Hv + h, (size_t)p.Hv, c1 - opub);
  }
}

// ---------------------------------------------------------------------------
// The output of chunk c for the value heads of key head kh on a whole CTA (`sm`:
// 1024-aligned, out_tc_smem bytes; `tmem`: 256 columns; lbar / mbar: the tiles' and the
// products' mbarriers with their running phases), value head by value head:
//   O = scale (diag(e^G) Q S + P Delta)
// in token rows, from the normalised Q tile of the key head (loaded once), the
// chunk-start state's S^T tile and the Delta^T tile the walk left, and P.  A head's tiles
// land while the previous head's epilogue runs.  Small enough (about 73 KB of shared
// memory, 256 TMEM columns, 48 registers) for two CTAs per SM, so that one CTA's loads
// and products also run under the other's epilogue.
__device__ void out_unit(const Params& p, int c, int kh, uint8_t* sm, uint32_t tmem,
                         uint64_t* lbar, uint32_t& ph, uint64_t* mbar, uint32_t& mph) {
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  const int Dk = p.Dk, Dv = p.Dv, MV = Dv < 64 ? 64 : Dv;
  const int tid = threadIdx.x, grp = col_group();
  const uint32_t bQ = (uint32_t)tileCD(Dk), bSt = tc::sw128_bytes(MV, Dk);
  const uint32_t bDt = (uint32_t)MV * 128, bP = 8192, bG = C * 4;
  uint8_t* tQ = sm;                  // [C][Dk] normalised Q of the key head
  uint8_t* tS = tQ + bQ;             // [MV][Dk] S^T
  uint8_t* tD = tS + bSt;            // [MV][C] Delta^T
  uint8_t* tP = tD + bDt;            // [C][C] P
  float* sG = (float*)(tP + bP);     // [C] G
  float* ev = sG + C;                // [C] scale e^G
  const uint32_t tO1 = tmem, tO2 = tmem + 128;   // Q S and P Delta (M = 64)
  const uint8_t* tiles = p.saved && p.bf16_states ? (const uint8_t*)p.saved : p.Stb;
  // thread 0: value head j's S^T, Delta^T, P and G tiles on one phase of bars[0]; for
  // KDA its own Q e^G tile instead of G (the key head's Q tile and e^G scaling serve the
  // scalar gate)
  auto issue_head = [&](int j, uint32_t extra) {
    const size_t ch = (size_t)c * p.Hv + value_head(p, kh, j);
    tc::mbar_arrive_expect_tx(lbar, extra + bSt + bDt + bP + (p.kda ? bQ : bG));
    tc::bulk_g2s(tS, tiles + ch * bSt, bSt, lbar);
    tc::bulk_g2s(tD, p.Dtb + ch * bDt, bDt, lbar);
    tc::bulk_g2s(tP, p.Psw + ch * bP, bP, lbar);
    if (p.kda)
      tc::bulk_g2s(tQ, p.Qgw + ch * bQ, bQ, lbar);
    else
      tc::bulk_g2s(sG, p.G + ch * C, bG, lbar);
  };
  if (tid == 0) {
    if (p.kda) {
      issue_head(0, 0u);
    } else {
      issue_head(0, bQ);
      tc::bulk_g2s(tQ, p.Qsw + ((size_t)c * p.Hk + kh) * bQ, bQ, lbar);
    }
  }
  for (int j = 0; j < p.r; ++j) {
    const int h = value_head(p, kh, j);
    const bool lok = tc::mbar_wait(lbar, ph);
    ph ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
      return;
    }
    if (tid < C) ev[tid] = p.kda ? p.scale : p.scale * expf(sG[tid]);
    // O1 = Q S (B = the S^T tile), O2 = P Delta (B = the Delta^T tile)
    const bool ok = mma_run([&] {
      tc::mma_tile_p(tO1, tc::smem_u32(tQ), 8192u, 64, tc::smem_u32(tS), (uint32_t)MV * 128u, Dv,
                     Dk, 0u);
      tc::mma_tile(tO2, tc::smem_u32(tP), 64, tc::smem_u32(tD), Dv, C, 0u);
    }, mbar, mph, p.status, c);
    if (!ok) return;
    // the products have read this head's tiles: the next head's land under the epilogue
    if (tid == 0 && j + 1 < p.r) issue_head(j + 1, 0u);
    // token row r of the chunk per accumulator lane, 16 consecutive values per thread (Dv
    // <= 128: one piece per thread; a row's pieces sit in the 8 threads of its lane pair in
    // the kGroups warps of its lane quarter)
    const int r = x2_row();
    const int col = grp * 16 + x2_half() * 16 * kGroups;
    const bool mine = r < len && col < Dv;
    __nv_bfloat16* orow = (__nv_bfloat16*)p.o + (t0 + r) * p.o_ld + (int64_t)h * Dv;
    float o1[16], o2[16];
    tc::tmem_ld16_x2<16 * kGroups>(tO1 + lane_quarter() + grp * 16, o1);
    tc::tmem_ld16_x2<16 * kGroups>(tO2 + lane_quarter() + grp * 16, o2);
    tc::tmem_ld_wait();
    __align__(16) __nv_bfloat162 pk[8];
    {
      const float e = ev[r];
  #pragma unroll
      for (int j = 0; j < 8; ++j)
        pk[j] = __floats2bfloat162_rn(fmaf(e, o1[2 * j], p.scale * o2[2 * j]),
                                      fmaf(e, o1[2 * j + 1], p.scale * o2[2 * j + 1]));
    }
    if (mine) {
      uint4* dst = (uint4*)(orow + col);
      dst[0] = ((const uint4*)pk)[0];
      dst[1] = ((const uint4*)pk)[1];
    }
    if (p.ny) {
      // gated RMSNorm of the row of o as stored (bf16): the sum of squares over the row's
      // pieces (lane pair, then the kGroups warps in a fixed order through shared memory)
      float* red = ev + C;   // [kGroups][C]
      float ss = 0.f;
      if (mine)
  #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = __bfloat1622float2(pk[j]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      ss = x2_pair_sum(ss);
      if (x2_half() == 0) red[grp * C + r] = ss;
      __syncthreads();
      float tot = 0.f;
  #pragma unroll
      for (int g = 0; g < kGroups; ++g) tot += red[g * C + r];
      if (mine) {
        const float inv = rsqrtf(fmaf(tot, 1.f / (float)Dv, p.neps));
        const __nv_bfloat16* zrow = (const __nv_bfloat16*)p.nz + (t0 + r) * p.nz_ld + (int64_t)h * Dv;
        const uint4 za = *(const uint4*)(zrow + col), zb = *(const uint4*)(zrow + col + 8);
        const __nv_bfloat162* z2[2] = {(const __nv_bfloat162*)&za, (const __nv_bfloat162*)&zb};
        __align__(16) __nv_bfloat162 yk[8];
  #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = __bfloat1622float2(pk[j]);
          const float2 z = __bfloat1622float2(z2[j >> 2][j & 3]);
          const float g0 = p.ngamma[col + 2 * j], g1 = p.ngamma[col + 2 * j + 1];
          yk[j] = __floats2bfloat162_rn(f.x * inv * g0 * (z.x * sigmoid_f(z.x)),
                                        f.y * inv * g1 * (z.y * sigmoid_f(z.y)));
        }
        uint4* ydst = (uint4*)((__nv_bfloat16*)p.ny + (t0 + r) * p.ny_ld + (int64_t)h * Dv + col);
        ydst[0] = ((const uint4*)yk)[0];
        ydst[1] = ((const uint4*)yk)[1];
      }
    }
  }
}

// The output pass: persistent CTAs (two per SM) take (chunk, key head) units from the
// output counter fwork[1] in chunk order; after a fused forward only the units it left.
__global__ void __launch_bounds__(kTcThreads, 2) k_fwd_out_tc(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  __shared__ int s_unit;
  cta_setup(ctl, 2, 256);
  const int ounits = p.NC * p.Hk;
  uint32_t lph = 0, mph = 0;
  int next = threadIdx.x == 0 ? (int)atomicAdd(p.fwork + 1, 1u) : 0;
  for (;;) {
    if (threadIdx.x == 0) s_unit = next;
    __syncthreads();
    const int u = s_unit;
    __syncthreads();
    if (u >= ounits) break;
    if (threadIdx.x == 0) next = (int)atomicAdd(p.fwork + 1, 1u);
    // one unit per (chunk, key head): the Q tile is loaded once for the group's heads
    out_unit(p, u / p.Hk, u % p.Hk, base + kCtlBytes, ctl->tmem, &ctl->bar[0], lph, &ctl->bar[1],
             mph);
  }
  cta_teardown(ctl, 256);
}

template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_fwd_state_tc(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  cta_setup(ctl, 4, 512);
  fwd_state_unit<DK, DV>(p, blockIdx.x, blockIdx.y, base + kCtlBytes, ctl->tmem, ctl->bar);
  cta_teardown(ctl, 512);
}

// The forward as one cooperative launch of one CTA per SM, for batches with fewer
// (sequence, value head) walks than SMs: CTAs [0, n_seqs * Hv) walk the chunks while
// the others prepare (chunk, key head) units in chunk order, taken from a work
// counter, and publish each one's flag; a walk waits for the flag of the chunk it
// needs next.  Walks never block the preparation, so the launch always finishes.
template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1) k_fwd_fused_tc(Params p,
                                                               const __grid_constant__ TmaMaps maps) {
  stamp_kept_operands(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  __shared__ int s_unit;
  cta_setup(ctl, 6, 512);
  const int walks = p.n_seqs * p.Hv;
  // Output units (chunk, key head) in chunk order from the second counter (fwork[1]),
  // each once its value heads' walks have published the chunk: the preparation CTAs take
  // them once the preparation is handed out, until the first walk finishes (fwork[2]
  // counts the finished walks; they finish within microseconds of each other), so that
  // the launch ends about when its walks do.  bar[4] / bar[5] serve them; neither role
  // used them before.  The output pass launched after this kernel takes the units left
  // (o and y are written by exactly one of them per unit).
  auto run_outputs = [&]() {
    const int ounits = p.oready ? p.NC * p.Hk : 0;
    uint32_t olph = 0, omph = 0;
    for (;;) {
      if (threadIdx.x == 0)
        s_unit = ld_relaxed(p.fwork + 2) == 0u ? (int)atomicAdd(p.fwork + 1, 1u) : ounits;
      __syncthreads();
      const int u = s_unit;
      __syncthreads();
      if (u >= ounits) break;
      const int c = u / p.Hk, kh = u % p.Hk;
      int bad = 0;
      for (int j = threadIdx.x; j < p.r; j += blockDim.x)
        if (!wait_flag(p.oready + (size_t)c * p.Hv + value_head(p, kh, j))) {
          set_status(p.status, GDN_ERR_TIMEOUT, c);
          bad = 1;
        }
      if (__syncthreads_or(bad)) break;
      if (threadIdx.x == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      out_unit(p, c, kh, base + kCtlBytes, ctl->tmem, &ctl->bar[4], olph, &ctl->bar[5], omph);
    }
  };
  if ((int)blockIdx.x < walks) {
    // One preparation unit first: the walk cannot start before the first chunk's units
    // are done anyway, so its CTA adds to the preparation's first wave.
    {
      const SeqTab tab =
          seq_tab(p, (int32_t*)(base + kCtlBytes + prep_buffers_bytes(p.Dk, p.Dv)), kSeqCache);
      if (threadIdx.x == 0) s_unit = (int)atomicAdd(p.fwork, 1u);
      __syncthreads();
      const int u = s_unit;
      if (u < p.NC * p.Hk) {
        uint32_t phase = 0, lphase = 0, vphase = 0;
        // every load and product of the unit has completed when it returns, and every
        // write came before its last barrier
        prep_unit<DK, DV>(p, maps, tab, p.keep, u / p.Hk, u % p.Hk, base + kCtlBytes, ctl->tmem,
                  ctl->bar, phase, lphase, vphase, nullptr);
        if (threadIdx.x == 0) {
          publish_flag(p.fready + u);
          // fresh mbarriers for the walk
          for (int i = 0; i < 4; ++i) {
            tc::mbar_inval(&ctl->bar[i]);
            tc::mbar_init(&ctl->bar[i], 1);
          }
          tc::fence_mbar_init();
        }
        __syncthreads();
      }
    }
    fwd_state_unit<DK, DV>(p, blockIdx.x / p.Hv, blockIdx.x % p.Hv, base + kCtlBytes, ctl->tmem,
                       ctl->bar);
    if (threadIdx.x == 0 && p.oready) atomicAdd(p.fwork + 2, 1u);
  } else {
    uint32_t phase = 0, lphase = 0, vphase = 0;
    const int units = p.NC * p.Hk;
    const SeqTab tab =
        seq_tab(p, (int32_t*)(base + kCtlBytes + prep_buffers_bytes(p.Dk, p.Dv)), kSeqCache);
    // the next unit is taken while the current one runs (thread 0's view); its value is
    // first read at the unit's last head, so the atomic's round trip stalls nobody
    PrepLink link{-1, -1, false};
    int next = threadIdx.x == 0 ? (int)atomicAdd(p.fwork, 1u) : 0;
    for (;;) {
      if (threadIdx.x == 0) s_unit = next;
      __syncthreads();
      const int u = s_unit;
      __syncthreads();
      if (u >= units) break;
      if (threadIdx.x == 0) {
        next = (int)atomicAdd(p.fwork, 1u);
        link.next = next;
      }
      const bool ok = prep_unit<DK, DV>(p, maps, tab, p.keep, u / p.Hk, u % p.Hk, base + kCtlBytes,
                                ctl->tmem, ctl->bar, phase, lphase, vphase, &link);
      if (threadIdx.x == 0) {
        if (link.pending >= 0) {   // a unit that stopped before its stores
          tc::bulk_wait<0>();
          publish_flag(p.fready + link.pending);
        }
        link.pending = u;
        // the first chunk's units are published at once: every walk starts with them
        if (u < p.Hk) {
          tc::bulk_wait<0>();
          publish_flag(p.fready + u);
          link.pending = -1;
        }
      }
      if (!ok) break;
    }
    if (threadIdx.x == 0) {
      // the last unit's stores, and k / q rows issued for a unit that will not run
      if (link.kq_issued) {
        tc::mbar_wait(&ctl->bar[1], lphase);
        tc::mbar_wait(&ctl->bar[2], vphase & 1u);
      }
      tc::bulk_wait<0>();
      if (link.pending >= 0) publish_flag(p.fready + link.pending);
    }
    run_outputs();
  }
  cta_teardown(ctl, 512);
}

// ---------------------------------------------------------------------------
static size_t prep_tc_smem(const Params& p) {
  return prep_buffers_bytes(p.Dk, p.Dv) + 2 * kSeqCache * sizeof(int32_t) + kCtlBytes + 1024;
}

static size_t out_tc_smem(const Params& p) {
  const int Dk = p.Dk, Dv = p.Dv, MV = Dv < 64 ? 64 : Dv;
  return tc::sw128_bytes(64, Dk) + tc::sw128_bytes(MV, Dk) + (size_t)MV * 128 + 8192 +
         (2 + kGroups) * C * 4 + kCtlBytes + 1024;
}

cudaError_t launch_fwd_out_tc(const Params& p, cudaStream_t st) {
  if (p.NC == 0) return cudaSuccess;
  const size_t smem = out_tc_smem(p);
  cudaFuncSetAttribute(k_fwd_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_FWD_OUT_TC);
  const int sms = sm_count();
  const int units = p.NC * p.Hk, grid = sms > 0 && 2 * sms < units ? 2 * sms : units;
  k_fwd_out_tc<<<(unsigned)grid, kTcThreads, smem, st>>>(p);
  profile_post(st);
  return cudaGetLastError();
}

template <int DK>
static size_t fwd_state_tc_smem(const Params& p) {
  const int Dv = p.Dv, MV = Dv < 64 ? 64 : Dv;
  const size_t bW = tc::sw128_bytes(64, DK);
  constexpr size_t EVS = DK > C ? DK : C;
  const size_t bU = (size_t)Dv * C * 2, bG = EVS * 4;
  const size_t bufsz = bW * 2 + ((bU + bG + 1023) & ~(size_t)1023);
  const size_t bHalf = ((size_t)(DK / 2) * Dv * 4 + 1023) & ~(size_t)1023;
  return tc::sw128_bytes(MV, DK) + 2 * bufsz + (size_t)MV * 128 + 2 * bHalf + 2 * EVS * 4 +
         kCtlBytes + 1024;
}

// The instantiations with the value head size fixed when it equals the key head size.
template <int DK>
static void (*prep_kernel(const Params& p))(Params, TmaMaps, int) {
  return p.Dv == DK ? k_prep_tc<DK, DK> : k_prep_tc<DK, 0>;
}

cudaError_t launch_prep_tc(const Params& p, const TmaMaps& maps, bool bwd, cudaStream_t st) {
  if (p.NC == 0) return cudaSuccess;
  const size_t smem = prep_tc_smem(p);
  auto kern = p.Dk == 128 ? prep_kernel<128>(p)
              : p.Dk == 64 ? prep_kernel<64>(p)
              : p.Dk == 32 ? prep_kernel<32>(p)
                           : prep_kernel<16>(p);
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, bwd ? KID_PREP_TC_FULL : KID_PREP_TC);
  kern<<<dim3(p.NC, p.Hk), kTcThreads, smem, st>>>(p, maps, bwd ? 1 : 0);
  profile_post(st);
  return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_fwd_state_tc_t(const Params& p, cudaStream_t st) {
  const size_t smem = fwd_state_tc_smem<DK>(p);
  auto kern = p.Dv == DK ? k_fwd_state_tc<DK, DK> : k_fwd_state_tc<DK, 0>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_FWD_STATE_TC);
  kern<<<dim3(p.n_seqs, p.Hv), kTcThreads, smem, st>>>(p);
  profile_post(st);
  return cudaGetLastError();
}

cudaError_t launch_fwd_state_tc(const Params& p, cudaStream_t st) {
  if (p.n_seqs == 0) return cudaSuccess;
  switch (p.Dk) {
    case 16: return launch_fwd_state_tc_t<16>(p, st);
    case 32: return launch_fwd_state_tc_t<32>(p, st);
    case 64: return launch_fwd_state_tc_t<64>(p, st);
    default: return launch_fwd_state_tc_t<128>(p, st);
  }
}

// The fused forward (k_fwd_fused_tc) when the walks leave at least kMinProducers SMs
// to the preparation and one CTA fits per SM; *launched = false otherwise (the caller
// then runs the preparation and the walk as two launches).
template <int DK, int DV>
static cudaError_t launch_fwd_fused_t(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                      bool* launched) {
  *launched = false;
  const int sms = sm_count();
  const int walks = p.n_seqs * p.Hv;
  if (sms <= 0 || walks + kMinProducers > sms || p.NC == 0) return cudaSuccess;
  const size_t a = prep_tc_smem(p), b = fwd_state_tc_smem<DK>(p);
  const size_t smem = (a > b ? a : b) + 64;
  cudaError_t e = cudaFuncSetAttribute(k_fwd_fused_tc<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fwd_fused_tc<DK, DV>, kTcThreads, smem);
  if (e != cudaSuccess || per_sm < 1) return cudaSuccess;
  Params pp = p;
  pp.fready = p.fwork + 64;             // the work counters' 256-byte slot, then the flags
  pp.oready = pp.fready + p.NC * p.Hk;  // the walks' chunk flags: the launch forms O too
  TmaMaps mm = maps;
  void* args[] = {&pp, &mm};
  profile_pre(st, KID_FWD_FUSED_TC);
  e = cudaLaunchCooperativeKernel((const void*)k_fwd_fused_tc<DK, DV>, dim3(sms), dim3(kTcThreads), args,
                                  smem, st);
  profile_post(st);
  if (e == cudaSuccess) *launched = true;
  return e;
}

template <int DK>
static cudaError_t launch_fwd_fused_dk(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                       bool* launched) {
  return p.Dv == DK ? launch_fwd_fused_t<DK, DK>(p, maps, st, launched)
                    : launch_fwd_fused_t<DK, 0>(p, maps, st, launched);
}

cudaError_t launch_fwd_fused_tc(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                bool* launched) {
  switch (p.Dk) {
    case 16: return launch_fwd_fused_dk<16>(p, maps, st, launched);
    case 32: return launch_fwd_fused_dk<32>(p, maps, st, launched);
    case 64: return launch_fwd_fused_dk<64>(p, maps, st, launched);
    default: return launch_fwd_fused_dk<128>(p, maps, st, launched);
  }
}

}  // namespace gdn
