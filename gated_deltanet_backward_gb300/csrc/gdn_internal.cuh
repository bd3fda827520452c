// gdn_internal.cuh -- shared declarations of the GB300 Gated DeltaNet kernels.
//
// Chunked form of the recurrence (derived from lattice-inference 0.6.0,
// gdn_backward.rs, module doc "Forward recap"; the pages name a chunked
// implementation, chunk_wy_forward_impl / ChunkWy::backward on the "KDA
// attention arm" work log, but do not write it out).  Per chunk of c <= 64
// tokens and value head h, rows r, s of the chunk:
//   l = log g, G = inclusive cumsum(l), E[r,s] = exp(G[r] - G[s]) (s <= r)
//   A = diag(b) (E * K K^T) strictly lower, T = (I + A)^-1
//   W = T diag(b e^G) K,  U = T diag(b) V,  Delta = U - W S
//   O = scale (diag(e^G) Q S + (E * Q K^T, lower) Delta)
//   S_next = e^{G[c-1]} S + K^T diag(e^{G[c-1] - G}) Delta
// K, Q are the L2-normalised keys / queries of key head h / v_repeat.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;     // tokens per chunk
constexpr int kThreads = 256;  // threads per CTA of every kernel

// Device-side status word layout at the start of the workspace.
struct DeviceStatus {
  int32_t code;    // first gdn_status recorded by a kernel (0 = OK)
  int32_t detail;  // kernel-specific detail (e.g. the chunk index)
  uint32_t tag;    // shape tag of a forward that kept the backward's operands (0 = none)
};

// Byte offsets of the workspace regions (fp32 unless noted; 0 = not allocated).
// C = 64 tokens per chunk; NC chunks.  fp32 inputs use the CUDA-core kernels'
// regions, bf16 inputs the tensor-core kernels' operand tiles (K-major,
// 128B-swizzled bf16, see umma.cuh), written by one kernel and copied as-is into
// shared memory by the next.
struct WsLayout {
  size_t status;  // DeviceStatus, 256 B
  size_t fsync;   // forward fused launch: work counters + (chunk, key head) and (chunk,
                  // value head) flags
  size_t bsync;   // backward fused launch: work counter + (chunk, value head) flags
  size_t nq;      // [NC][Hk][C] query norms sqrt(|q|^2 + 1e-6)
  size_t nk;      // [NC][Hk][C] key norms
  size_t G;       // [NC][Hv][C] inclusive cumsum of log g
  size_t b;       // [NC][Hv][C] beta
  size_t pa;      // [NC][Hv] per-chunk partial of d a_log (backward)
  size_t pd;      // [NC][Hv] per-chunk partial of d dt_bias (backward)
  // fp32 path
  size_t Qn;      // [NC][Hk][C][Dk] normalised queries
  size_t Kn;      // [NC][Hk][C][Dk] normalised keys
  size_t W;       // [NC][Hv][C][Dk]
  size_t U;       // [NC][Hv][C][Dv]
  size_t Tm;      // [NC][Hv][C][C] (backward)
  size_t dS;      // [NC][Hv][Dk][Dv] state adjoint at each chunk end (backward)
  size_t dD;      // [NC][Hv][C][Dv] d Delta (backward)
  size_t dQh;     // [NC][Hv][C][Dk] per-value-head d q_hat partials (backward)
  size_t dKh;     // [NC][Hv][C][Dk] per-value-head d k_hat partials (backward)
  // bf16 path (tiles)
  // (a product that wants one of these transposed reads it MN-major)
  size_t Qsw;     // [NC][Hk] [C][Dk]   normalised queries
  size_t Ksw;     // [NC][Hk] [C][Dk]   normalised keys
  size_t Wsw;     // [NC][Hv] [C][Dk]   W
  size_t Psw;     // [NC][Hv] [C][C]    P = E * (Q K^T), lower incl. diagonal
  size_t Utb;     // [NC][Hv] [Dv][C]   U^T
  size_t KKf;     // [NC][Hk][C][C] fp32  K K^T (backward)
  size_t Tb;      // [NC][Hv] 2 x [C][C]: T, T diag(b e^G) (backward)
  size_t dSb;     // [NC][Hv] [MV][Dk] dS^T: state adjoint at each chunk end (backward)
  size_t dDb;     // [NC][Hv] [C][MV]  -d Delta (backward); MV = max(Dv, 64)
  size_t Stb;     // [NC][Hv] [MV][Dk] S^T: chunk-start states as bf16 operand tiles, written
                  // by the walk for the output pass (and kept for a reusing backward)
  size_t Dtb;     // [NC][Hv] [MV][C] Delta^T, written by the walk for the output pass
  size_t Kcw;     // [NC][Hv] [C][Dk]   diag(e^{G_last - G}) K, the state update's operand
  size_t total;
};

// Bytes of the bf16 SW128 operand tiles (C = 64 rows or columns).
inline size_t tile_CxD(int D) { return (size_t)((D + 63) / 64) * 64 * 128; }
inline size_t tile_DxD(int R, int D) { return (size_t)((D + 63) / 64) * R * 128; }
// Bytes of one bf16 state tile: S^T (or dS^T) with max(Dv, 64) rows and Dk columns.
inline size_t state_tile_bytes(int Dk, int Dv) { return tile_DxD(Dv < 64 ? 64 : Dv, Dk); }

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline WsLayout ws_layout(const gdn_shape& s, bool bwd) {
  WsLayout L{};
  const size_t NC = (size_t)s.total_chunks, C = kChunk;
  const size_t Hk = s.Hk, Hv = s.Hv, Dk = s.Dk, Dv = s.Dv;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L.status = take(256);
  // readiness flags of the fused launches, right after the status block so that one
  // memset clears both: forward [256 B: preparation and output work counters | NC*Hk
  // preparation flags | NC*Hv walk flags], backward [256 B work counter | NC*Hv flags]
  L.fsync = take(256 + NC * Hk * 4 + NC * Hv * 4);
  L.bsync = take(256 + NC * Hv * 4);
  L.nq = take(NC * Hk * C * 4);
  L.nk = take(NC * Hk * C * 4);
  L.G = take(NC * Hv * C * 4);
  L.b = take(NC * Hv * C * 4);
  if (bwd) {
    L.pa = take(NC * Hv * 4);
    L.pd = take(NC * Hv * 4);
  }
  if (s.dtype != GDN_DTYPE_BF16) {
    L.Qn = take(NC * Hk * C * Dk * 4);
    L.Kn = take(NC * Hk * C * Dk * 4);
    L.W = take(NC * Hv * C * Dk * 4);
    L.U = take(NC * Hv * C * Dv * 4);
    if (bwd) {
      L.Tm = take(NC * Hv * C * C * 4);
      L.dS = take(NC * Hv * Dk * Dv * 4);
      L.dD = take(NC * Hv * C * Dv * 4);
      L.dQh = take(NC * Hv * C * Dk * 4);
      L.dKh = take(NC * Hv * C * Dk * 4);
    }
  } else {
    L.Qsw = take(NC * Hk * tile_CxD(s.Dk));
    L.Ksw = take(NC * Hk * tile_CxD(s.Dk));
    L.Wsw = take(NC * Hv * tile_CxD(s.Dk));
    L.Psw = take(NC * Hv * tile_CxD(64));
    L.Utb = take(NC * Hv * Dv * C * 2);
    L.Stb = take(NC * Hv * state_tile_bytes(s.Dk, s.Dv));
    L.Dtb = take(NC * Hv * (size_t)(Dv < 64 ? 64 : Dv) * 128);
    L.Kcw = take(NC * Hv * tile_CxD(s.Dk));
    if (bwd) {
      L.KKf = take(NC * Hk * C * C * 4);
      L.Tb = take(NC * Hv * 2 * tile_CxD(64));
      L.dSb = take(NC * Hv * state_tile_bytes(s.Dk, s.Dv));
      L.dDb = take(NC * Hv * tile_CxD(s.Dv));
    }
  }
  L.total = off;
  return L;
}

// Everything a kernel needs, passed by value.
struct Params {
  int Hk, Hv, Dk, Dv, r, n_seqs, NC;
  int head_map;  // 0: key head h / r; 1: key head h % Hk
  int64_t T;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  int64_t q_ld, k_ld, v_ld;
  const float* alpha;
  const float* beta_raw;
  int64_t alpha_ld, beta_ld;
  const float* a_log;
  const float* dt_bias;
  const int32_t* cu;
  const int32_t* coff;
  const float* S0;
  void* o;
  int64_t o_ld;
  float* S_T;
  float* saved;
  const float* saved_in;
  const void* dO;
  int64_t dO_ld;
  const float* dS_T;
  void* dq;
  void* dk;
  void* dv;
  int64_t dq_ld, dk_ld, dv_ld;
  float* dalpha;
  float* dbeta;
  int64_t dalpha_ld, dbeta_ld;
  float* da_log;
  float* ddt_bias;
  float* dS0;
  DeviceStatus* status;
  uint32_t* fwork;   // fused forward: next preparation unit; fwork[1]: next output unit
  uint32_t* fready;  // fused forward: [NC][Hk] preparation unit done
  uint32_t* oready;  // fused forward: [NC][Hv] the walk's S^T and Delta^T tiles of the
                     // chunk stored (the output units read them); null: no output units
  uint32_t* bwork;   // fused backward: next gradient unit
  uint32_t* bready;  // fused backward: [NC][Hv] state-walk chunk done
  uint32_t tag;  // shape tag (see shape_tag); written by a keeping forward, checked by a reusing backward
  // forward with the gated RMSNorm of o fused into its output pass (ny null: none):
  // y = (o / sqrt(mean o^2 + neps)) * ngamma * SiLU(z) per (token, value head) row
  const void* nz;
  int64_t nz_ld;
  const float* ngamma;
  float neps;
  void* ny;
  int64_t ny_ld;
  int keep;      // forward: leave the backward's chunk operands in the workspace
  int bf16_states;  // chunk-start states as bf16 S^T tiles (GDN_FLAG_BF16_SAVED_STATES)
                    // instead of fp32 [NC][Hv][Dk][Dv]
  int reuse;     // backward: read them from the workspace instead of recomputing them
  float* Qn;
  float* Kn;
  float* nq;
  float* nk;
  float* W;
  float* U;
  float* Tm;
  float* G;
  float* b;
  float* dS;
  float* dD;
  float* dQh;
  float* dKh;
  float* pa;
  float* pd;
  uint8_t* Qsw;
  uint8_t* Ksw;
  uint8_t* Wsw;
  uint8_t* Psw;
  __nv_bfloat16* Utb;
  float* KKf;
  uint8_t* Tb;
  uint8_t* dSb;
  uint8_t* dDb;
  uint8_t* Stb;
  uint8_t* Dtb;
  uint8_t* Kcw;
  // chunked KDA forward (a decay gate per key channel): kda set, the gates from alpha
  // [T, Hv*Dk] and b_alpha [Hv*Dk]; its preparation leaves per (chunk, value head) the
  // tile Q * e^G (Qgw, [C][Dk], the output's operand) and e^{G_last} (Gl, [Dk], the
  // walk's per-channel decay); the walk and the output pass read those instead of G
  int kda;
  const float* b_alpha;
  uint8_t* Qgw;
  float* Gl;
};

// Key head of value head h, and the j-th (j < r) value head of key head kh: value
// heads h and h' share a key head when h / r == h' / r (head_map 0, consecutive) or
// h % Hk == h' % Hk (head_map 1, modulo).
__host__ __device__ __forceinline__ int key_head(const Params& p, int h) {
  return p.head_map ? h % p.Hk : h / p.r;
}
__host__ __device__ __forceinline__ int value_head(const Params& p, int kh, int j) {
  return p.head_map ? kh + j * p.Hk : kh * p.r + j;
}

// Kernel ids reported to the profiling hook (gdn_profile_begin).
enum KernelId {
  KID_PREP = 0,
  KID_FWD_STATE = 1,
  KID_BWD_STATE = 2,
  KID_BWD_GRADS = 3,
  KID_BWD_QK = 4,
  KID_BWD_GATES = 5,
  KID_PREP_TC = 6,
  KID_FWD_STATE_TC = 7,
  KID_BWD_STATE_TC = 8,
  KID_BWD_GRADS_TC = 9,
  KID_PREP_TC_FULL = 10,
  KID_FWD_FUSED_TC = 11,
  KID_BWD_FUSED_TC = 12,
  KID_DECODE = 13,
  KID_CONV_FWD = 14,
  KID_CONV_BWD = 15,
  KID_NORM_FWD = 16,
  KID_NORM_BWD = 17,
  KID_SUM_PARTS = 18,
  KID_COMPOSE = 19,
  KID_KDA_FWD = 20,
  KID_KDA_BWD = 21,
  KID_FWD_OUT_TC = 22,
  KID_KDA_PREP_TC = 23,
  KID_COUNT = 24
};

// Bracket one launch with the caller's profiling events (no-op when none are
// registered on this host thread).
void profile_pre(cudaStream_t st, int kernel_id);
void profile_post(cudaStream_t st);

// TMA tensor maps of the bf16 row-major inputs: 2-D (columns, tokens), boxes of
// 64 columns x 64 tokens, 128-byte swizzle (the K-major SW128 operand layout),
// out-of-range rows and columns read as zero.
struct TmaMaps {
  CUtensorMap q, k, v, dO;
};

// Encodes `m` over a [rows, ld] bf16 matrix of which the first `cols` columns are
// used.  Returns false if the driver rejects it.
bool encode_tma_2d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld);

// Tensor-core (bf16) launchers.
cudaError_t launch_prep_tc(const Params& p, const TmaMaps& maps, bool bwd, cudaStream_t st);
// Fused launches need a producer CTA beside the walks on at least this many SMs.
constexpr int kMinProducers = 8;
// SMs of the current device (cached per device; 0 if the query fails).
int sm_count();
cudaError_t launch_fwd_fused_tc(const Params& p, const TmaMaps& maps, cudaStream_t st,
                                bool* launched);
cudaError_t launch_fwd_state_tc(const Params& p, cudaStream_t st);
// The output pass of the bf16 forward: O from the walk's state and Delta tiles.
cudaError_t launch_fwd_out_tc(const Params& p, cudaStream_t st);
cudaError_t launch_kda_prep_tc(const Params& p, const TmaMaps& maps, cudaStream_t st);
cudaError_t launch_bwd_tc(const Params& p, const TmaMaps& maps, cudaStream_t st);

// One decode step (gdn_decode_step): arguments validated by the caller.
// Causal depthwise conv1d + SiLU and gated RMSNorm (gdn_neighbours.cu).  `part` is the
// caller's scratch for the weight gradient's per-block partial sums (conv_partial_floats /
// norm_partial_floats floats); dw / dgamma null skips them.
size_t conv_partial_floats(int64_t T, int C, int K);
size_t norm_partial_floats(int D);
cudaError_t launch_conv1d_silu(bool bwd, int dtype, int64_t T, int C, int K, const int32_t* cu,
                               int n_seqs, const void* x, int64_t x_ld, const float* w,
                               const void* dy, int64_t dy_ld, void* y, int64_t y_ld, float* dw,
                               float* part, cudaStream_t st);
cudaError_t launch_gated_rmsnorm(bool bwd, int dtype, int64_t T, int H, int D, float eps,
                                 const void* o, int64_t o_ld, const void* z, int64_t z_ld,
                                 const float* gamma, const void* dy, int64_t dy_ld, void* y,
                                 int64_t y_ld, void* dz, int64_t dz_ld, float* dgamma,
                                 float* part, cudaStream_t st);
// out = op(Phi) S + R for n blocks (gdn_context.cu); R may be null (zero).
cudaError_t launch_state_compose(int n, int Dk, int Dv, const float* Phi, const float* S,
                                 const float* R, float* out, bool transpose, cudaStream_t st);
// The KDA variant's token-form forward (gdn_kda.cu).
cudaError_t launch_kda_forward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                               int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                               int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                               const float* a_log, const float* b_alpha, const int32_t* cu,
                               const float* S_in, float* S_out, void* o, int64_t o_ld,
                               cudaStream_t st);
// Its backward (gdn_kda.cu): saved states, per-slice shares and sums in `ws`
// (kda_bwd_workspace_floats floats).
size_t kda_bwd_workspace_floats(const gdn_shape* s);
cudaError_t launch_kda_backward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                                int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                                int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                                const float* a_log, const float* b_alpha, const int32_t* cu,
                                const float* S0, const void* dO, int64_t dO_ld,
                                const float* dS_T, void* dq, int64_t dq_ld, void* dk,
                                int64_t dk_ld, void* dv, int64_t dv_ld, float* dalpha,
                                int64_t dalpha_ld, float* dbeta, int64_t dbeta_ld, float* da_log,
                                float* db_alpha, float* dS0, float* ws, cudaStream_t st);
cudaError_t launch_decode(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                          int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                          int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                          const float* a_log, const float* dt_bias, const float* S_in,
                          float* S_out, void* o, int64_t o_ld, cudaStream_t st);

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_prep(const Params& p, bool write_T, cudaStream_t st);
cudaError_t launch_forward(const Params& p, const TmaMaps* maps, cudaStream_t st);
cudaError_t launch_backward(const Params& p, const TmaMaps* maps, cudaStream_t st);

}  // namespace gdn
