// gdn_tc_kda.cu -- the chunk preparation of the KDA variant (a decay gate per key channel)
// on the tensor cores: k_kda_prep_tc, one CTA per (chunk, value head).  The chunk walk and
// the output pass that consume its tiles are the scalar-gate ones of gdn_tc_fwd.cu with a
// per-channel decay (Params::kda).  Notation as in gdn_internal.cuh; every product is
// D = A B^T with A, B K-major.
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int C = kChunk;
constexpr int TS = C + 4;   // row stride (floats) of the fp32 [C][C] matrices of the inverse

// Thread 0: the raw k and q rows of key head kh of the chunk at token t0 as TMA boxes into
// the [K; Q] tile (K rows 0-63, Q rows 64-127 of each 64-column block), on one phase of
// `bar`.
__device__ void load_kq_rows(const Params& p, const TmaMaps& maps, int64_t t0, int kh,
                             uint8_t* tAQK, uint64_t* bar) {
  const int nbk = (p.Dk + 63) / 64;
  tc::mbar_arrive_expect_tx(bar, 2u * nbk * 8192u);
  for (int b = 0; b < nbk; ++b) {
    tc::tma_load_2d(tAQK + b * 128 * 128, &maps.k, kh * p.Dk + 64 * b, (int)t0, bar);
    tc::tma_load_2d(tAQK + b * 128 * 128 + 8192, &maps.q, kh * p.Dk + 64 * b, (int)t0, bar);
  }
}

// T = (I + A)^-1 of one head (Tm: A strictly lower on entry, T on return; M: a
// 1024-float scratch) on threads 0-255, which meet on named barrier 1: 16x16 diagonal
// blocks by substitution, then the 32x32 and the 64x64 lower-left blocks as
// -D_1 A_10 D_0 (2x2 block inversion at two levels), every product spread over all 256
// threads in 1 x 2 or 1 x 4 pieces.
__device__ void tri_inverse_one_head(float* Tm, float* M) {
  const int tid = threadIdx.x;
  const auto sync = [] { asm volatile("bar.sync 1, 256;" ::: "memory"); };
  // 16x16 diagonal blocks, thread j of block b solving column j column-wise: once x_k is
  // final it updates every later row, so the dependent chain is 16 FMAs long
  {
    const int b = tid >> 4, j = tid & 15;
    float* B = Tm + (tid < 64 ? b * (16 * TS + 16) : 0);
    float x[16];
    if (tid < 64) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int k = 0; k < 15; ++k) {
        float col[15];
#pragma unroll
        for (int i = k + 1; i < 16; ++i) col[i - 1] = B[i * TS + k];
#pragma unroll
        for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-col[i - 1], x[k], x[i]);
      }
    }
    sync();
    if (tid < 64)
#pragma unroll
      for (int i = 0; i < 16; ++i) B[i * TS + j] = x[i];
    sync();
  }
  // 32x32 diagonal blocks (rows / columns 32 q .. 32 q + 31): M = A_10 D_0, then
  // A_10 <- -D_1 M; thread: block q, row r, columns c0, c0 + 1.  Every load of a product
  // is issued before its FMAs.
  {
    const int q = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
    const int cb = 32 * q, rb = cb + 16;
    float a[16];
    float2 d[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      a[k] = Tm[(rb + r) * TS + cb + k];
      d[k] = *(const float2*)(Tm + (cb + k) * TS + cb + c0);
    }
    float m0 = 0.f, m1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      m0 = fmaf(a[k], d[k].x, m0);
      m1 = fmaf(a[k], d[k].y, m1);
    }
    *(float2*)(M + q * 256 + r * 16 + c0) = make_float2(m0, m1);
    sync();
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      a[k] = Tm[(rb + r) * TS + rb + k];
      d[k] = *(const float2*)(M + q * 256 + k * 16 + c0);
    }
    float t0 = 0.f, t1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      t0 = fmaf(a[k], d[k].x, t0);
      t1 = fmaf(a[k], d[k].y, t1);
    }
    *(float2*)(Tm + (rb + r) * TS + cb + c0) = make_float2(-t0, -t1);
    sync();
  }
  // 64x64: M = A_BA T_A, then A_BA <- -T_B M; thread: row r, columns c0 .. c0 + 3, eight
  // k steps of loads at a time
  {
    const int r = tid >> 3, c0 = (tid & 7) * 4;
    const auto product = [&](const float* rowp, const float* colp, int ld) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k0 = 0; k0 < 32; k0 += 8) {
        float a[8];
        float4 t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          a[u] = rowp[k0 + u];
          t[u] = *(const float4*)(colp + (k0 + u) * ld);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc.x = fmaf(a[u], t[u].x, acc.x);
          acc.y = fmaf(a[u], t[u].y, acc.y);
          acc.z = fmaf(a[u], t[u].z, acc.z);
          acc.w = fmaf(a[u], t[u].w, acc.w);
        }
      }
      return acc;
    };
    *(float4*)(M + r * 32 + c0) = product(Tm + (32 + r) * TS, Tm + c0, TS);
    sync();
    const float4 acc = product(Tm + (32 + r) * TS + 32, M + c0, 32);
    *(float4*)(Tm + (32 + r) * TS + c0) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    sync();
  }
}

// KDA variant (a decay gate per key channel, the KDA work log's module gate): one (chunk
// c, value head h) preparation unit on a whole CTA (`sm`: 1024-aligned, kda_prep_bytes;
// `tmem`: 256 columns; bar[0..2]: products, k / q rows, V rows).  The chunk algebra of
// the per-channel recurrence, per value head (its gates differ from head to head):
//   l[r][i] = -e^{a_log[h]} softplus(alpha[t][h Dk + i] + b_alpha[h Dk + i]),
//   G = inclusive cumsum of l over the chunk's rows, channel by channel,
//   A[r][s] = b_r sum_i K[r][i] K[s][i] e^{G[r][i] - G[s][i]}   (s < r),
//   P[r][s] =     sum_i Q[r][i] K[s][i] e^{G[r][i] - G[s][i]}   (s <= r).
// G does not increase along the rows, so a pair's exponent is <= 0, but neither e^G nor
// e^{-G} alone stays in range when the gates decay fast.  The rows fall into four blocks
// of 16, and each block j takes its first row 16 j as a reference: for r in block j and
// any s <= r, G[r] - G[s] = (G[r] - G[16 j]) + (G[16 j] - G[s]), so block j's rows of A
// and P are one product on the tensor core of the rows X[r] e^{G[r] - G[16 j]} (X = K
// or Q; exponent <= 0) with K[s] e^{G[16 j] - G[s]} (s < 16 j + 16).  Before the block
// the second exponent is <= 0 as well; inside it, it is at most the block's decay
// G[16 j] - G[16 j + 15], so the block's own pairs come from the product only where
// that stays below kKdaWide for every channel (e^60 keeps the operand, and the masked
// entries above the diagonal, far from overflow and the block's own factor
// e^{G[r] - G[16 j]} far from underflow).  A block whose gates decay faster zeroes those
// rows of the operand and sums its 136 pairs channel by channel on CUDA cores, eight
// threads a pair, every exponent <= 0.
// Then T = (I + A)^-1, W = T diag(b) (K e^G) and U^T = V^T (T diag(b))^T on the tensor
// core, and the operands of the walk and the output: K e^{G_last - G} (the state
// update), Q e^G (the output's inter-chunk term), e^{G_last} (the walk's per-channel
// decay) and P.  Rows past the chunk are zero and take no decay.  Dk, Dv in {64, 128}.
constexpr int kGS = 128 + 4;   // row stride (floats) of the fp32 [C][Dk] gate matrix
constexpr int kKdaBlk = 16;    // rows of a block of the intra-chunk products
constexpr float kKdaWide = 60.f;   // largest in-block decay taken through the product

// softplus with the hardware exp2 / log2 approximations: log(1 + e^x) for x <= 15 (the
// sum 1 + e^x then stays exact to fp32 rounding), x above.  Its absolute error stays
// near 1e-6 (the log's), against gates of order 1 that the chunk only ever sums and
// exponentiates.
__device__ __forceinline__ float softplus_approx(float x) {
  return x > 15.f ? x : __logf(1.f + __expf(x));
}

__host__ __device__ __forceinline__ size_t kda_prep_bytes(int Dk, int Dv) {
  const size_t nbk = (size_t)(Dk + 63) / 64, nbv = (size_t)(Dv + 63) / 64;
  return nbk * 128 * 128 + nbv * 8192 + 2 * 8192 + nbk * 8192 + nbk * 160 * 128 +
         sizeof(float) * ((size_t)C * kGS + (size_t)C * TS + 1024 + C + 4);
}

template <int DK>
__device__ void kda_prep_unit(const Params& p, const TmaMaps& maps, int c, int h, uint8_t* sm,
                              uint32_t tmem, uint64_t* bar) {
  int n;
  int64_t t0;
  int len;
  if (!chunk_info(p, c, &n, &t0, &len)) {
    if (threadIdx.x == 0) set_status(p.status, GDN_ERR_DEVICE_BOUNDS, c);
    return;
  }
  constexpr int Dk = DK, NK = DK, nbk = (DK + 63) / 64;
  const int Dv = p.Dv, MV = Dv;
  const int tid = threadIdx.x, kh = key_head(p, h);
  const int nbv = (Dv + 63) / 64;
  const uint32_t aqk_pitch = 128u * 128u, bKC = tc::sw128_bytes(64, Dk);
  uint8_t* tAQK = sm;                          // [128][Dk]: rows 0-63 K, 64-127 Q
  uint8_t* sV = tAQK + nbk * aqk_pitch;        // [C][Dv] natural V (TMA)
  uint8_t* tTB = sV + nbv * 8192;              // [C][C] T diag(b)
  uint8_t* tP = tTB + 8192;                    // [C][C] P
  uint8_t* tKg = tP + 8192;                    // [C][Dk] K e^G
  // [128][Dk] block-scaled K; Q rows of the intra-chunk products, over tTB .. tKg (which
  // are written only after those products)
  uint8_t* tXs = tTB;
  uint8_t* tKn = tKg + bKC;                    // [160][Dk] block-scaled K (block j from row
                                               // 8 j (j + 1) on)
  float* Gf = (float*)(tKn + nbk * 160 * 128); // [C][kGS] G
  float* Tm = Gf + C * kGS;                    // [C][TS] A, then T
  float* Mt = Tm + C * TS;                     // [1024] diagonal blocks of P, then the
                                               // inverse's scratch
  float* bv = Mt + 1024;                       // [C] beta
  int* wide = (int*)(bv + C);                  // [4] block decays faster than kKdaWide
  const uint32_t tAccW = tmem, tAccU = tmem + 128;
  const size_t ch = (size_t)c * p.Hv + h;
  uint32_t phase = 0, lphase = 0, vphase = 0;
  if (tid == 0) {
    load_kq_rows(p, maps, t0, kh, tAQK, &bar[1]);
    tc::mbar_arrive_expect_tx(&bar[2], (uint32_t)nbv * 8192u);
    for (int b = 0; b < nbv; ++b)
      tc::tma_load_2d(sV + b * 8192, &maps.v, h * Dv + 64 * b, (int)t0, &bar[2]);
  }
  // 1. the gate inputs (a thread's alpha loads all in flight at once: channel gi of the
  // kRpt rows from gr0 on) and beta; A starts at zero
  constexpr int kRpt = C * Dk / kTcThreads;   // 16 (Dk = 128) or 8 (Dk = 64)
  const int gi = tid % Dk, gpart = tid / Dk, gr0 = gpart * kRpt;
  float av[kRpt];
  {
    const float* arow = p.alpha + (size_t)h * Dk + gi;
#pragma unroll
    for (int u = 0; u < kRpt; ++u)
      av[u] = gr0 + u < len ? arow[(t0 + gr0 + u) * p.alpha_ld] : 0.f;
    if (tid < C) bv[tid] = tid < len ? sigmoid_f(p.beta_raw[(t0 + tid) * p.beta_ld + h]) : 0.f;
    if (tid < 4) wide[tid] = 0;
    for (int i2 = tid; i2 < C * TS; i2 += kTcThreads) Tm[i2] = 0.f;
  }
  // 2. L2 normalisation of the k / q rows in place (four threads per row), rows past the
  // chunk zero, while the gate loads land
  {
    const bool lok = tc::mbar_wait(&bar[1], lphase);
    lphase ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
      return;
    }
  }
  {
    const int row = tid >> 2, part = tid & 3, t = row & (C - 1);
    constexpr int nch = Dk / 8, cpt = nch / 4;
    uint4 raw[cpt];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < cpt; ++j) {
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
    const float inv = t < len ? 1.f / sqrtf(ss + 1e-6f) : 0.f;
#pragma unroll
    for (int j = 0; j < cpt; ++j) {
      const __nv_bfloat162* e = (const __nv_bfloat162*)&raw[j];
      __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(e[q]);
        pk[q] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
      }
      *(uint4*)(tAQK + tc::sw128_offset(row, (part * cpt + j) * 8, 128)) = *(const uint4*)pk;
    }
  }
  // 3. l and its cumsum over the rows: each thread sums its own rows in registers, then
  // adds the totals of the rows before them (through Mt); the blocks' decays
  {
    const float ea = expf(p.a_log[h]);
    const float ba = p.b_alpha[(size_t)h * Dk + gi];
    float run = 0.f;
#pragma unroll
    for (int u = 0; u < kRpt; ++u) {
      run += gr0 + u < len ? -ea * softplus_approx(av[u] + ba) : 0.f;
      av[u] = run;
    }
    Mt[gpart * Dk + gi] = run;
    __syncthreads();
    float off = 0.f;
    for (int q = 0; q < gpart; ++q) off += Mt[q * Dk + gi];
#pragma unroll
    for (int u = 0; u < kRpt; ++u) Gf[(gr0 + u) * kGS + gi] = off + av[u];
    constexpr int kPpb = kKdaBlk / kRpt;   // threads (row ranges) per block of 16 rows
    if (gpart % kPpb == 0) {
      float decay = 0.f;
#pragma unroll
      for (int q = 0; q < kPpb; ++q) decay -= Mt[(gpart + q) * Dk + gi];
      if (decay > kKdaWide) wide[gpart / kPpb] = 1;
    }
  }
  __syncthreads();
  // 4. A and P.  Row r of tXs (K rows 0-63, Q rows 64-127) is X[r] e^{G[r] - G[16 j(r)]};
  // rows 8 j (j+1) .. 8 (j+1) (j+2) - 1 of tKn hold K[s] e^{G[16 j] - G[s]} for s < 16 j + 16
  // (the last 16 of them zero when block j is wide), so one product of N = 160 forms every
  // block's columns.
  // Four channels a thread (a warp reads a G row as one contiguous 512-byte line); the
  // factor e^{G[s] - G[ref]} of a tXs row serves its K and its Q row.  A pass of the CTA
  // covers kRowsPass rows, so the tXs rows take the first kXsPasses passes and the tKn
  // rows the rest, for every thread alike (compile-time trip counts, unrolled).
  {
    constexpr int c4n = Dk / 4, kRowsPass = kTcThreads / c4n;
    constexpr int kXsPasses = C / kRowsPass, kKnPasses = 160 / kRowsPass;
    const int k4 = (tid % c4n) * 4, prow = tid / c4n;
#pragma unroll
    for (int it = 0; it < kXsPasses; ++it) {
      const int s = prow + it * kRowsPass, gref = (s / kKdaBlk) * kKdaBlk;
      const float4 gs = *(const float4*)(Gf + s * kGS + k4);
      const float4 gr = *(const float4*)(Gf + gref * kGS + k4);
      const uint2 kraw = *(const uint2*)(tAQK + tc::sw128_offset(s, k4, 128));
      const uint2 qraw = *(const uint2*)(tAQK + tc::sw128_offset(C + s, k4, 128));
      const float e0 = __expf(gs.x - gr.x), e1 = __expf(gs.y - gr.y);
      const float e2 = __expf(gs.z - gr.z), e3 = __expf(gs.w - gr.w);
      const __nv_bfloat162* k2 = (const __nv_bfloat162*)&kraw;
      const __nv_bfloat162* q2 = (const __nv_bfloat162*)&qraw;
      const float2 k01 = __bfloat1622float2(k2[0]), k23 = __bfloat1622float2(k2[1]);
      const float2 q01 = __bfloat1622float2(q2[0]), q23 = __bfloat1622float2(q2[1]);
      __align__(8) __nv_bfloat162 ok2[2], oq2[2];
      ok2[0] = __floats2bfloat162_rn(k01.x * e0, k01.y * e1);
      ok2[1] = __floats2bfloat162_rn(k23.x * e2, k23.y * e3);
      oq2[0] = __floats2bfloat162_rn(q01.x * e0, q01.y * e1);
      oq2[1] = __floats2bfloat162_rn(q23.x * e2, q23.y * e3);
      *(uint2*)(tXs + tc::sw128_offset(s, k4, 128)) = *(const uint2*)ok2;
      *(uint2*)(tXs + tc::sw128_offset(C + s, k4, 128)) = *(const uint2*)oq2;
    }
#pragma unroll
    for (int it = 0; it < kKnPasses; ++it) {
      const int q = prow + it * kRowsPass;   // tKn row: block j = 0..3 of 16 (j + 1) rows
      const int j = q < 16 ? 0 : (q < 48 ? 1 : (q < 96 ? 2 : 3));
      const int s = q - 8 * j * (j + 1), gref = j * kKdaBlk;
      const bool zero = s >= gref && wide[j];
      const float4 gs = *(const float4*)(Gf + s * kGS + k4);
      const float4 gr = *(const float4*)(Gf + gref * kGS + k4);
      const uint2 kraw = *(const uint2*)(tAQK + tc::sw128_offset(s, k4, 128));
      const __nv_bfloat162* k2 = (const __nv_bfloat162*)&kraw;
      const float2 k01 = __bfloat1622float2(k2[0]), k23 = __bfloat1622float2(k2[1]);
      const float e0 = zero ? 0.f : __expf(gr.x - gs.x), e1 = zero ? 0.f : __expf(gr.y - gs.y);
      const float e2 = zero ? 0.f : __expf(gr.z - gs.z), e3 = zero ? 0.f : __expf(gr.w - gs.w);
      __align__(8) __nv_bfloat162 o2[2];
      o2[0] = __floats2bfloat162_rn(k01.x * e0, k01.y * e1);
      o2[1] = __floats2bfloat162_rn(k23.x * e2, k23.y * e3);
      *(uint2*)(tKn + tc::sw128_offset(q, k4, 160)) = *(const uint2*)o2;
    }
  }
  tc::fence_async_smem();
  mma_issue([&] {
    tc::mma_tile_p(tmem, tc::smem_u32(tXs), 128u * 128u, 128, tc::smem_u32(tKn), 160u * 128u,
                   160, Dk, 0u);
  }, &bar[0]);
  // wide blocks: their pairs s <= r, eight threads a pair (each 1/8 of the channels): A
  // into Tm, P into the [4][16][16] diagonal-block scratch Mt.  A warp's four pairs lie
  // in one block.
  const int nwide = wide[0] + wide[1] + wide[2] + wide[3];
  for (int idx = tid; nwide != 0 && idx < 4 * 136 * 8; idx += kTcThreads) {
    const int pr = idx >> 3, part = idx & 7, blk = pr / 136, t = pr % 136;
    if (!wide[blk]) continue;
    int rr = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
    while ((rr + 1) * (rr + 2) / 2 <= t) ++rr;
    while (rr * (rr + 1) / 2 > t) --rr;
    const int ss = t - rr * (rr + 1) / 2;
    const int r = blk * kKdaBlk + rr, s = blk * kKdaBlk + ss;
    float a = 0.f, pp = 0.f;
    for (int k8 = part * 8; k8 < Dk; k8 += 64) {
      const uint4 kr = *(const uint4*)(tAQK + tc::sw128_offset(r, k8, 128));
      const uint4 ks = *(const uint4*)(tAQK + tc::sw128_offset(s, k8, 128));
      const uint4 qr = *(const uint4*)(tAQK + tc::sw128_offset(C + r, k8, 128));
      const float* gr = Gf + r * kGS + k8;
      const float* gs = Gf + s * kGS + k8;
      const float4 ga = *(const float4*)gr, gb = *(const float4*)(gr + 4);
      const float4 ha = *(const float4*)gs, hb = *(const float4*)(gs + 4);
      const float e[8] = {__expf(ga.x - ha.x), __expf(ga.y - ha.y), __expf(ga.z - ha.z),
                          __expf(ga.w - ha.w), __expf(gb.x - hb.x), __expf(gb.y - hb.y),
                          __expf(gb.z - hb.z), __expf(gb.w - hb.w)};
      const __nv_bfloat162* k2r = (const __nv_bfloat162*)&kr;
      const __nv_bfloat162* k2s = (const __nv_bfloat162*)&ks;
      const __nv_bfloat162* q2r = (const __nv_bfloat162*)&qr;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 fr = __bfloat1622float2(k2r[q]), fs = __bfloat1622float2(k2s[q]);
        const float2 fq = __bfloat1622float2(q2r[q]);
        const float k0 = fs.x * e[2 * q], k1 = fs.y * e[2 * q + 1];
        a = fmaf(fr.x, k0, fmaf(fr.y, k1, a));
        pp = fmaf(fq.x, k0, fmaf(fq.y, k1, pp));
      }
    }
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, d);
      pp += __shfl_xor_sync(0xffffffffu, pp, d);
    }
    if (part == 0) {
      if (ss < rr) Tm[r * TS + s] = bv[r] * a;
      Mt[blk * 256 + rr * 16 + ss] = pp;
    }
  }
  if (!mma_wait(&bar[0], phase, p.status, c)) return;
  // accumulator columns [8 j (j+1), 8 (j+1) (j+2)) hold block j's rows against s < 16 j +
  // 16; a lane row (K rows, then Q rows) takes the 16-column pieces of its own block,
  // masked to s < r (A) or s <= r (P) on the diagonal, which a wide block leaves out
  acc_walk(tmem, 128, 160, 128, [&](int row, int col0, const float* v) {
    const int r = row & (C - 1), j = r / kKdaBlk;
    const int pj = col0 < 16 ? 0 : (col0 < 48 ? 1 : (col0 < 96 ? 2 : 3));
    if (pj != j) return;
    const int s0 = col0 - 8 * j * (j + 1);
    const bool diag = s0 == j * kKdaBlk;
    if (diag && wide[j]) return;
    if (row < C) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (!diag || s0 + e < r) Tm[r * TS + s0 + e] = bv[r] * v[e];
    } else {
      float m[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) m[e] = (!diag || s0 + e <= r) ? v[e] : 0.f;
      tile_put16(tP, C, r, s0, m);
    }
  });
  // the rest of P: the diagonal blocks of wide blocks from the scratch, zeros above the
  // diagonal blocks
  for (int idx = tid; idx < C * (C / 8); idx += kTcThreads) {
    const int r = idx >> 3, c8 = (idx & 7) * 8, j = r / kKdaBlk, bc = c8 / kKdaBlk;
    if (bc < j || (bc == j && !wide[j])) continue;
    __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float x0 = 0.f, x1 = 0.f;
      if (bc == j) {
        const int s = c8 + 2 * u;
        const float* pd = Mt + j * 256 + (r % kKdaBlk) * 16 + (s % kKdaBlk);
        x0 = s <= r ? pd[0] : 0.f;
        x1 = s + 1 <= r ? pd[1] : 0.f;
      }
      pk[u] = __floats2bfloat162_rn(x0, x1);
    }
    *(uint4*)(tP + tc::sw128_offset(r, c8, C)) = *(const uint4*)pk;
  }
  __syncthreads();
  // 5. T = (I + A)^-1 on warps 0-7, while the other warps write the operands that do not
  // need T: P, Q e^G, K e^{G_last - G} and e^{G_last} into the workspace, K e^G into its
  // product tile (four channels a thread)
  if (tid < 256) {
    tri_inverse_one_head(Tm, Mt);
  } else {
    constexpr int nt2 = kTcThreads - 256, c4n = NK / 4;
    const int t2 = tid - 256;
#pragma unroll
    for (int i = t2; i < C * (C / 8); i += nt2) {
      const uint32_t off = tc::sw128_offset(i >> 3, (i & 7) * 8, C);
      *(uint4*)(p.Psw + ch * 8192 + off) = *(const uint4*)(tP + off);
    }
    const float* gl = Gf + (len - 1) * kGS;
    const int k4 = (t2 % c4n) * 4;
#pragma unroll 4
    for (int s = t2 / c4n; s < C; s += nt2 / c4n) {
      const float4 g = *(const float4*)(Gf + s * kGS + k4);
      const float4 gL = *(const float4*)(gl + k4);
      const uint2 kraw = *(const uint2*)(tAQK + tc::sw128_offset(s, k4, 128));
      const uint2 qraw = *(const uint2*)(tAQK + tc::sw128_offset(C + s, k4, 128));
      const __nv_bfloat162* k2 = (const __nv_bfloat162*)&kraw;
      const __nv_bfloat162* q2 = (const __nv_bfloat162*)&qraw;
      const float e[4] = {__expf(g.x), __expf(g.y), __expf(g.z), __expf(g.w)};
      const bool in = s < len;
      const float cd[4] = {in ? __expf(gL.x - g.x) : 0.f, in ? __expf(gL.y - g.y) : 0.f,
                           in ? __expf(gL.z - g.z) : 0.f, in ? __expf(gL.w - g.w) : 0.f};
      __align__(8) __nv_bfloat162 kg[2], qg[2], kc[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float2 fk = __bfloat1622float2(k2[q]), fq = __bfloat1622float2(q2[q]);
        kg[q] = __floats2bfloat162_rn(fk.x * e[2 * q], fk.y * e[2 * q + 1]);
        qg[q] = __floats2bfloat162_rn(fq.x * e[2 * q], fq.y * e[2 * q + 1]);
        kc[q] = __floats2bfloat162_rn(fk.x * cd[2 * q], fk.y * cd[2 * q + 1]);
      }
      const uint32_t off = tc::sw128_offset(s, k4, C);
      *(uint2*)(tKg + off) = *(const uint2*)kg;
      *(uint2*)(p.Qgw + ch * bKC + off) = *(const uint2*)qg;
      *(uint2*)(p.Kcw + ch * bKC + off) = *(const uint2*)kc;
    }
    if (t2 < Dk) p.Gl[ch * Dk + t2] = expf(gl[t2]);
  }
  __syncthreads();
  // 6. T diag(b) into its product tile
  {
    const int r = tid >> 3, s8 = (tid & 7) * 8;   // one 8-column piece of T a thread
    __align__(16) __nv_bfloat162 pb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      pb[u] = __floats2bfloat162_rn(Tm[r * TS + s8 + 2 * u] * bv[s8 + 2 * u],
                                    Tm[r * TS + s8 + 2 * u + 1] * bv[s8 + 2 * u + 1]);
    *(uint4*)(tTB + tc::sw128_offset(r, s8, C)) = *(const uint4*)pb;
  }
  // 7. V rows (past the chunk zero), then W = T diag(b) (K e^G) and U^T = V^T (T diag(b))^T
  {
    const bool lok = tc::mbar_wait(&bar[2], vphase & 1u);
    vphase ^= 1u;
    if (__syncthreads_or(lok ? 0 : 1)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT, c);
      return;
    }
  }
  if (len < C)
    for (int idx = tid; idx < nbv * (C - len) * 8; idx += kTcThreads) {
      const int b2 = idx / ((C - len) * 8), rem = idx % ((C - len) * 8);
      ((uint4*)(sV + b2 * 8192 + (len + rem / 8) * 128))[rem % 8] = make_uint4(0, 0, 0, 0);
    }
  tc::fence_async_smem();
  const bool ok = mma_run([&] {
    // W = (T diag(b)) (K e^G): B is K e^G read MN-major from its natural tile
    tc::mma_tile_x(tAccW, tc::smem_u32(tTB), false, 8192u, 64, tc::smem_u32(tKg), true, 8192u,
                   NK, C, 0u);
    // U^T = V^T (T diag(b))^T: A is V^T read MN-major from the natural V tile
    tc::mma_tile_x(tAccU, tc::smem_u32(sV), true, 8192u, MV, tc::smem_u32(tTB), false, 8192u, C,
                   C, 0u);
  }, &bar[0], phase, p.status, c);
  if (!ok) return;
  acc_walk64(tAccW, Dk, C, [&](int s, int col0, const float* v) {
    tile_put16(p.Wsw + ch * bKC, C, s, col0, v);
  });
  acc_walk(tAccU, MV, 64, Dv, [&](int vv, int col0, const float* v) {
    tile_put16((uint8_t*)(p.Utb + ch * Dv * C), Dv, vv, col0, v);
  });
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

template <int DK>
__global__ void __launch_bounds__(kTcThreads, 1) k_kda_prep_tc(Params p,
                                                              const __grid_constant__ TmaMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  CtaCtl* ctl = (CtaCtl*)base;
  cta_setup(ctl, 3, 256);
  kda_prep_unit<DK>(p, maps, blockIdx.x, blockIdx.y, base + kCtlBytes, ctl->tmem, ctl->bar);
  cta_teardown(ctl, 256);
}

}  // namespace

cudaError_t launch_kda_prep_tc(const Params& p, const TmaMaps& maps, cudaStream_t st) {
  if (p.NC == 0) return cudaSuccess;
  const size_t smem = kda_prep_bytes(p.Dk, p.Dv) + kCtlBytes + 1024;
  auto kern = p.Dk == 128 ? k_kda_prep_tc<128> : k_kda_prep_tc<64>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  profile_pre(st, KID_KDA_PREP_TC);
  kern<<<dim3(p.NC, p.Hv), kTcThreads, smem, st>>>(p, maps);
  profile_post(st);
  return cudaGetLastError();
}

}  // namespace gdn
