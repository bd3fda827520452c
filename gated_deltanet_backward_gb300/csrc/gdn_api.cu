// gdn_api.cu -- the C ABI of libgdn.so: argument checks, workspace carving and
// kernel launches.  See include/gdn.h for the contract of every entry point.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"

using gdn::Params;
using gdn::WsLayout;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool head_size_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

int check_shape(const gdn_shape* s) {
  if (!s) return GDN_ERR_INVALID_ARG;
  if (s->Hk <= 0 || s->Hv <= 0 || s->n_seqs < 0 || s->total_tokens < 0 || s->total_chunks < 0)
    return GDN_ERR_INVALID_ARG;
  if (s->Hv % s->Hk != 0) return GDN_ERR_INVALID_ARG;
  if (!head_size_ok(s->Dk) || !head_size_ok(s->Dv)) return GDN_ERR_UNSUPPORTED;
  if (s->dtype != GDN_DTYPE_F32 && s->dtype != GDN_DTYPE_BF16) return GDN_ERR_UNSUPPORTED;
  if (s->head_map != GDN_HEAD_MAP_CONSECUTIVE && s->head_map != GDN_HEAD_MAP_MODULO)
    return GDN_ERR_INVALID_ARG;
  if (!(s->scale >= 0.f) || std::isinf(s->scale)) return GDN_ERR_INVALID_ARG;
  // a chunk holds at least one token, and every token lies in some chunk
  if ((int64_t)s->total_chunks > s->total_tokens) return GDN_ERR_INVALID_ARG;
  if ((int64_t)s->total_chunks * gdn::kChunk < s->total_tokens) return GDN_ERR_INVALID_ARG;
  if (s->n_seqs == 0 && s->total_tokens != 0) return GDN_ERR_INVALID_ARG;
  // grid limits of the per-chunk kernels
  if (s->total_chunks > 0x3fffffff || s->Hv > 65535 || s->n_seqs > 0x3fffffff)
    return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// A dtype-typed matrix argument [total_tokens, ld] holding `width` used columns.
int check_matrix(const void* p, int64_t ld, int64_t width, size_t esize, int64_t rows) {
  if (rows == 0) return GDN_OK;
  if (!p) return GDN_ERR_INVALID_ARG;
  if (ld < width) return GDN_ERR_INVALID_ARG;
  if (!aligned16(p) || ((size_t)ld * esize) % 16 != 0) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

// An fp32 per-head matrix [total_tokens, ld] (alpha, beta_raw and their grads).
int check_gate_matrix(const void* p, int64_t ld, int64_t Hv, int64_t rows) {
  if (rows == 0) return GDN_OK;
  if (!p) return GDN_ERR_INVALID_ARG;
  if (ld < Hv) return GDN_ERR_INVALID_ARG;
  if (((uintptr_t)p & 3u) != 0) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

int check_vec(const void* p, bool required) {
  if (!p) return required ? GDN_ERR_INVALID_ARG : GDN_OK;
  if (!aligned16(p)) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

// An fp32 per-head vector (a_log, dt_bias and their gradients): read and written one
// element at a time, so 4-byte alignment (a sub-vector of one rank's heads passes).
int check_head_vec(const void* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (((uintptr_t)p & 3u) != 0) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

// Byte ranges of two [rows, ld] matrices (width used columns) intersect.
bool overlaps(const void* a, int64_t a_ld, const void* b, int64_t b_ld, int64_t rows,
              int64_t width, size_t esize) {
  if (!a || !b || rows == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  const uintptr_t a1 = a0 + ((size_t)(rows - 1) * a_ld + width) * esize;
  const uintptr_t b1 = b0 + ((size_t)(rows - 1) * b_ld + width) * esize;
  return a0 < b1 && b0 < a1;
}

int check_dtype(int32_t dtype, size_t* esize) {
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_UNSUPPORTED;
  *esize = dtype == GDN_DTYPE_BF16 ? 2 : 4;
  return GDN_OK;
}

int check_scratch(const void* ws, size_t bytes, size_t need) {
  if (need == 0) return GDN_OK;
  if (!ws || bytes < need) return GDN_ERR_WORKSPACE;
  if (!aligned16(ws)) return GDN_ERR_WORKSPACE;
  return GDN_OK;
}

#define GDN_TRY(x)                 \
  do {                             \
    const int _rc = (x);           \
    if (_rc != GDN_OK) return _rc; \
  } while (0)

int check_conv(int32_t dtype, int64_t T, int32_t C, int32_t K, const int32_t* cu, int32_t n_seqs,
               const float* w, size_t* es) {
  GDN_TRY(check_dtype(dtype, es));
  if (T < 0 || C <= 0 || n_seqs < 0 || (T > 0 && n_seqs == 0)) return GDN_ERR_INVALID_ARG;
  if (K < 1 || K > 4 || C % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (T > (int64_t)1 << 30 || C > 1 << 24) return GDN_ERR_UNSUPPORTED;  // 32-bit tile indices
  if (T > 0 && !cu) return GDN_ERR_INVALID_ARG;
  if (cu && ((uintptr_t)cu & 3u) != 0) return GDN_ERR_MISALIGNED;
  return check_vec(w, true);
}

int check_norm(int32_t dtype, int64_t T, int32_t H, int32_t D, float eps, const float* gamma,
               size_t* es) {
  GDN_TRY(check_dtype(dtype, es));
  if (T < 0 || H <= 0 || !(eps >= 0.f) || eps > 3.0e38f) return GDN_ERR_INVALID_ARG;
  if (!head_size_ok(D)) return GDN_ERR_UNSUPPORTED;
  if (T * H * (int64_t)D > (int64_t)1 << 31) return GDN_ERR_UNSUPPORTED;  // 32-bit vector indices
  return check_vec(gamma, true);
}

void fill_common(Params& p, const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                 int64_t k_ld, const void* v, int64_t v_ld, const float* alpha, int64_t alpha_ld,
                 const float* beta_raw, int64_t beta_ld, const float* a_log, const float* dt_bias,
                 const int32_t* cu, const int32_t* coff, const float* S0, void* ws, bool bwd) {
  std::memset(&p, 0, sizeof(p));
  p.Hk = s->Hk;
  p.Hv = s->Hv;
  p.Dk = s->Dk;
  p.Dv = s->Dv;
  p.r = s->Hv / s->Hk;
  p.head_map = s->head_map;
  p.n_seqs = s->n_seqs;
  p.NC = s->total_chunks;
  p.T = s->total_tokens;
  p.scale = s->scale > 0.f ? s->scale : 1.0f / std::sqrt((float)s->Dk);
  p.q = q;
  p.k = k;
  p.v = v;
  p.q_ld = q_ld;
  p.k_ld = k_ld;
  p.v_ld = v_ld;
  p.alpha = alpha;
  p.beta_raw = beta_raw;
  p.alpha_ld = alpha_ld;
  p.beta_ld = beta_ld;
  p.a_log = a_log;
  p.dt_bias = dt_bias;
  p.cu = cu;
  p.coff = coff;
  p.S0 = S0;
  const WsLayout L = gdn::ws_layout(*s, bwd);
  char* base = (char*)ws;
  p.status = (gdn::DeviceStatus*)(base + L.status);
  // flag arrays are handed to the kernels only by the fused launchers
  p.fwork = (uint32_t*)(base + L.fsync);
  p.fready = nullptr;
  p.oready = nullptr;
  p.bwork = (uint32_t*)(base + L.bsync);
  p.bready = nullptr;
  p.nq = (float*)(base + L.nq);
  p.nk = (float*)(base + L.nk);
  p.G = (float*)(base + L.G);
  p.b = (float*)(base + L.b);
  if (bwd) {
    p.pa = (float*)(base + L.pa);
    p.pd = (float*)(base + L.pd);
  }
  if (s->dtype != GDN_DTYPE_BF16) {
    p.Qn = (float*)(base + L.Qn);
    p.Kn = (float*)(base + L.Kn);
    p.W = (float*)(base + L.W);
    p.U = (float*)(base + L.U);
    if (bwd) {
      p.Tm = (float*)(base + L.Tm);
      p.dS = (float*)(base + L.dS);
      p.dD = (float*)(base + L.dD);
      p.dQh = (float*)(base + L.dQh);
      p.dKh = (float*)(base + L.dKh);
    }
  } else {
    p.Qsw = (uint8_t*)(base + L.Qsw);
    p.Ksw = (uint8_t*)(base + L.Ksw);
    p.Wsw = (uint8_t*)(base + L.Wsw);
    p.Psw = (uint8_t*)(base + L.Psw);
    p.Utb = (__nv_bfloat16*)(base + L.Utb);
    p.Stb = (uint8_t*)(base + L.Stb);
    p.Dtb = (uint8_t*)(base + L.Dtb);
    p.Kcw = (uint8_t*)(base + L.Kcw);
    if (bwd) {
      p.KKf = (float*)(base + L.KKf);
      p.Tb = (uint8_t*)(base + L.Tb);
      p.dSb = (uint8_t*)(base + L.dSb);
      p.dDb = (uint8_t*)(base + L.dDb);
    }
  }
}

int check_inputs(const gdn_shape* s, const void* q, int64_t q_ld, const void* k, int64_t k_ld,
                 const void* v, int64_t v_ld, const float* alpha, int64_t alpha_ld,
                 const float* beta_raw, int64_t beta_ld, const float* a_log,
                 const float* dt_bias, const int32_t* cu, const int32_t* coff, const float* S0) {
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int64_t T = s->total_tokens;
  GDN_TRY(check_matrix(q, q_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(k, k_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(v, v_ld, (int64_t)s->Hv * s->Dv, es, T));
  GDN_TRY(check_gate_matrix(alpha, alpha_ld, s->Hv, T));
  GDN_TRY(check_gate_matrix(beta_raw, beta_ld, s->Hv, T));
  GDN_TRY(check_head_vec(a_log));
  GDN_TRY(check_head_vec(dt_bias));
  if (!cu || !coff) return GDN_ERR_INVALID_ARG;
  if (((uintptr_t)cu & 3u) || ((uintptr_t)coff & 3u)) return GDN_ERR_MISALIGNED;
  GDN_TRY(check_vec(S0, false));
  return GDN_OK;
}

int check_workspace(const gdn_shape* s, void* ws, size_t bytes, bool bwd) {
  if (!ws) return GDN_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return GDN_ERR_WORKSPACE;
  if (bytes < gdn::ws_layout(*s, bwd).total) return GDN_ERR_WORKSPACE;
  return GDN_OK;
}

// Tag of a shape (FNV-1a over its fields, never 0): a keeping forward stamps it
// into the workspace's status block and a reusing backward compares it.
uint32_t shape_tag(const gdn_shape* s) {
  const int64_t f[9] = {s->Hk, s->Hv, s->Dk, s->Dv, s->n_seqs, s->total_chunks, s->total_tokens,
                        s->dtype, s->head_map};
  uint32_t h = 2166136261u;
  auto mix = [&](const void* data, size_t n) {
    const unsigned char* b = (const unsigned char*)data;
    for (size_t i = 0; i < n; ++i) h = (h ^ b[i]) * 16777619u;
  };
  mix(f, sizeof(int64_t) * 9);
  mix(&s->scale, sizeof(float));
  return h | 1u;
}

thread_local char g_last_error[160] = "";

// Records which CUDA call failed (see gdn_last_error) and returns GDN_ERR_CUDA.
int cuda_fail(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return GDN_ERR_CUDA;
}

struct ProfileState {
  void* const* events = nullptr;
  int32_t* ids = nullptr;
  int32_t n_pairs = 0;
  int32_t count = 0;
  bool on = false;
};
thread_local ProfileState g_profile;

}  // namespace

namespace gdn {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}
}  // namespace

bool encode_tma_2d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0, coop = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop)
      cached[dev] = n;
    else
      cached[dev] = -1;
  }
  return cached[dev] > 0 ? cached[dev] : 0;
}

// Lets other translation units of the library explain a failure through
// gdn_last_error().
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

void profile_pre(cudaStream_t st, int kernel_id) {
  ProfileState& P = g_profile;
  if (!P.on) return;
  if (P.count < P.n_pairs) {
    P.ids[P.count] = kernel_id;
    cudaEventRecord((cudaEvent_t)P.events[2 * P.count], st);
  }
}

void profile_post(cudaStream_t st) {
  ProfileState& P = g_profile;
  if (!P.on) return;
  if (P.count < P.n_pairs) cudaEventRecord((cudaEvent_t)P.events[2 * P.count + 1], st);
  ++P.count;
}

}  // namespace gdn

extern "C" {

int gdn_profile_begin(void* const* events, int32_t* kernel_ids, int32_t n_pairs) {
  if (n_pairs < 0 || (n_pairs > 0 && (!events || !kernel_ids))) return GDN_ERR_INVALID_ARG;
  g_profile.events = events;
  g_profile.ids = kernel_ids;
  g_profile.n_pairs = n_pairs;
  g_profile.count = 0;
  g_profile.on = true;
  return GDN_OK;
}

int gdn_profile_end(void) {
  const int n = g_profile.count;
  g_profile = ProfileState();
  return n;
}

const char* gdn_last_error(void) { return g_last_error; }

const char* gdn_kernel_name(int32_t id) {
  switch (id) {
    case gdn::KID_PREP: return "gdn_prep";
    case gdn::KID_FWD_STATE: return "gdn_fwd_state";
    case gdn::KID_BWD_STATE: return "gdn_bwd_state";
    case gdn::KID_BWD_GRADS: return "gdn_bwd_grads";
    case gdn::KID_BWD_QK: return "gdn_bwd_qk";
    case gdn::KID_BWD_GATES: return "gdn_bwd_gates";
    case gdn::KID_PREP_TC: return "gdn_prep_tc";
    case gdn::KID_FWD_STATE_TC: return "gdn_fwd_state_tc";
    case gdn::KID_BWD_STATE_TC: return "gdn_bwd_state_tc";
    case gdn::KID_BWD_GRADS_TC: return "gdn_bwd_grads_tc";
    case gdn::KID_PREP_TC_FULL: return "gdn_prep_tc_full";
    case gdn::KID_FWD_FUSED_TC: return "gdn_fwd_fused_tc";
    case gdn::KID_BWD_FUSED_TC: return "gdn_bwd_fused_tc";
    case gdn::KID_DECODE: return "gdn_decode";
    case gdn::KID_CONV_FWD: return "gdn_conv1d_silu_fwd";
    case gdn::KID_CONV_BWD: return "gdn_conv1d_silu_bwd";
    case gdn::KID_NORM_FWD: return "gdn_gated_rmsnorm_fwd";
    case gdn::KID_NORM_BWD: return "gdn_gated_rmsnorm_bwd";
    case gdn::KID_SUM_PARTS: return "gdn_sum_partials";
    case gdn::KID_COMPOSE: return "gdn_state_compose";
    case gdn::KID_KDA_FWD: return "gdn_kda_fwd";
    case gdn::KID_KDA_BWD: return "gdn_kda_bwd";
    case gdn::KID_FWD_OUT_TC: return "gdn_fwd_out_tc";
    case gdn::KID_KDA_PREP_TC: return "gdn_kda_prep_tc";
    default: return "?";
  }
}

int gdn_plan(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t* chunk_offsets_host,
             int32_t* total_chunks) {
  if (!cu_seqlens_host || !chunk_offsets_host || !total_chunks || n_seqs < 0)
    return GDN_ERR_INVALID_ARG;
  if (cu_seqlens_host[0] != 0) return GDN_ERR_INVALID_ARG;
  int64_t acc = 0;
  chunk_offsets_host[0] = 0;
  for (int32_t n = 0; n < n_seqs; ++n) {
    const int64_t len = (int64_t)cu_seqlens_host[n + 1] - cu_seqlens_host[n];
    if (len < 0) return GDN_ERR_INVALID_ARG;
    acc += (len + gdn::kChunk - 1) / gdn::kChunk;
    if (acc > 0x3fffffff) return GDN_ERR_INVALID_ARG;
    chunk_offsets_host[n + 1] = (int32_t)acc;
  }
  *total_chunks = (int32_t)acc;
  return GDN_OK;
}

size_t gdn_saved_state_bytes(const gdn_shape* s) {
  if (check_shape(s) != GDN_OK) return 0;
  return (size_t)s->total_chunks * s->Hv * s->Dk * s->Dv * sizeof(float);
}

namespace {
// GDN_FLAG_BF16_SAVED_STATES: bf16 inputs with Dk, Dv >= 64 (so that the bf16 tiles,
// padded to 64 rows and columns, fit in the fp32 buffer's bytes).
int check_bf16_states(const gdn_shape* s, uint32_t flags, int* on) {
  *on = (flags & GDN_FLAG_BF16_SAVED_STATES) != 0;
  if (*on && (s->dtype != GDN_DTYPE_BF16 || s->Dk < 64 || s->Dv < 64)) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}
// The shape tag a keeping forward leaves and a reusing backward checks, covering the
// saved states' format too.
uint32_t keep_tag(const gdn_shape* s, int bf16_states) {
  return bf16_states ? (shape_tag(s) ^ 0x5bd1e994u) | 1u : shape_tag(s);
}
}  // namespace

size_t gdn_workspace_bytes(const gdn_shape* s, int is_backward) {
  if (check_shape(s) != GDN_OK) return 0;
  return gdn::ws_layout(*s, is_backward != 0).total;
}

// The gated RMSNorm that a forward may apply to its own output (y null: none).
struct FwdNorm {
  const void* z = nullptr;
  int64_t z_ld = 0;
  const float* gamma = nullptr;
  float eps = 0.f;
  void* y = nullptr;
  int64_t y_ld = 0;
};

static int forward_impl(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                        int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                        int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                        const float* a_log, const float* dt_bias, const int32_t* cu_seqlens,
                        const int32_t* chunk_offsets, const float* S0, void* o, int64_t o_ld,
                        float* S_T, void* saved_states, void* workspace, size_t workspace_bytes,
                        uint32_t flags, const FwdNorm& nm, void* stream) {
  GDN_TRY(check_shape(s));
  if (flags & ~(uint32_t)(GDN_FLAG_KEEP_FOR_BACKWARD | GDN_FLAG_BF16_SAVED_STATES))
    return GDN_ERR_INVALID_ARG;
  const bool keep = (flags & GDN_FLAG_KEEP_FOR_BACKWARD) != 0;
  int bf16_states = 0;
  GDN_TRY(check_bf16_states(s, flags, &bf16_states));
  GDN_TRY(check_inputs(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                       dt_bias, cu_seqlens, chunk_offsets, S0));
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  GDN_TRY(check_matrix(o, o_ld, (int64_t)s->Hv * s->Dv, es, s->total_tokens));
  if (nm.y) {
    const int64_t T = s->total_tokens, W = (int64_t)s->Hv * s->Dv;
    size_t nes = 0;
    GDN_TRY(check_norm(s->dtype, T, s->Hv, s->Dv, nm.eps, nm.gamma, &nes));
    GDN_TRY(check_matrix(nm.z, nm.z_ld, W, es, T));
    GDN_TRY(check_matrix(nm.y, nm.y_ld, W, es, T));
    if (overlaps(o, o_ld, nm.y, nm.y_ld, T, W, es) || overlaps(nm.z, nm.z_ld, nm.y, nm.y_ld, T, W, es) ||
        overlaps(o, o_ld, nm.z, nm.z_ld, T, W, es))
      return GDN_ERR_INVALID_ARG;
  }
  GDN_TRY(check_vec(S_T, false));
  // a forward that no backward reads (prefill, inference) may skip the saved states
  GDN_TRY(check_vec(saved_states, keep && s->total_chunks > 0));
  GDN_TRY(check_workspace(s, workspace, workspace_bytes, keep));
  cudaStream_t st = (cudaStream_t)stream;
  Params p;
  // a keeping forward carves the backward's layout, whose forward regions sit
  // at the same offsets as the backward will read them
  fill_common(p, s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
              dt_bias, cu_seqlens, chunk_offsets, S0, workspace, keep);
  p.keep = keep ? 1 : 0;
  p.bf16_states = bf16_states;
  p.tag = keep_tag(s, bf16_states);
  p.o = o;
  p.o_ld = o_ld;
  p.S_T = S_T;
  p.saved = (float*)saved_states;
  (void)cudaGetLastError();  // report only errors of this call's own launches
  g_last_error[0] = 0;
  // status block and the fused forward's flags (they follow it)
  const gdn::WsLayout L = gdn::ws_layout(*s, keep);
  cudaError_t e = cudaMemsetAsync(workspace, 0, L.bsync, st);
  if (e != cudaSuccess) return cuda_fail("gdn_forward: clearing the status word", e);
  if (s->n_seqs > 0 && s->total_chunks == 0) {
    // every sequence is empty: S_T = S_0
    if (!S_T) return GDN_OK;
    const size_t bytes = (size_t)s->n_seqs * s->Hv * s->Dk * s->Dv * sizeof(float);
    e = S0 ? cudaMemcpyAsync(S_T, S0, bytes, cudaMemcpyDeviceToDevice, st)
           : cudaMemsetAsync(S_T, 0, bytes, st);
    return e == cudaSuccess ? GDN_OK : cuda_fail("gdn_forward: S_T of empty sequences", e);
  }
  gdn::TmaMaps maps;
  const bool bf16 = s->dtype == GDN_DTYPE_BF16;
  if (bf16 && s->total_tokens > 0) {
    const int64_t T = s->total_tokens;
    if (!gdn::encode_tma_2d(&maps.q, q, (int64_t)s->Hk * s->Dk, T, q_ld) ||
        !gdn::encode_tma_2d(&maps.k, k, (int64_t)s->Hk * s->Dk, T, k_ld) ||
        !gdn::encode_tma_2d(&maps.v, v, (int64_t)s->Hv * s->Dv, T, v_ld)) {
      snprintf(g_last_error, sizeof(g_last_error), "gdn_forward: cuTensorMapEncodeTiled failed");
      return GDN_ERR_CUDA;
    }
  }
  if (nm.y && bf16) {
    // bf16: the output pass normalises the rows it forms
    p.nz = nm.z;
    p.nz_ld = nm.z_ld;
    p.ngamma = nm.gamma;
    p.neps = nm.eps;
    p.ny = nm.y;
    p.ny_ld = nm.y_ld;
  }
  e = gdn::launch_forward(p, bf16 ? &maps : nullptr, st);
  if (e != cudaSuccess) return cuda_fail("gdn_forward: kernel launch", e);
  if (nm.y && !bf16 && s->total_tokens > 0) {
    e = gdn::launch_gated_rmsnorm(false, s->dtype, s->total_tokens, s->Hv, s->Dv, nm.eps, o, o_ld,
                                  nm.z, nm.z_ld, nm.gamma, nullptr, 0, nm.y, nm.y_ld, nullptr, 0,
                                  nullptr, nullptr, st);
    if (e != cudaSuccess) return cuda_fail("gdn_forward_gated_rmsnorm: norm launch", e);
  }
  return GDN_OK;
}

int gdn_forward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k, int64_t k_ld,
                const void* v, int64_t v_ld, const float* alpha, int64_t alpha_ld,
                const float* beta_raw, int64_t beta_ld, const float* a_log,
                const float* dt_bias, const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                const float* S0, void* o, int64_t o_ld, float* S_T, void* saved_states,
                void* workspace, size_t workspace_bytes, uint32_t flags, void* stream) {
  return forward_impl(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                      dt_bias, cu_seqlens, chunk_offsets, S0, o, o_ld, S_T, saved_states,
                      workspace, workspace_bytes, flags, FwdNorm(), stream);
}

int gdn_forward_gated_rmsnorm(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                              int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                              int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                              const float* a_log, const float* dt_bias,
                              const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                              const float* S0, void* o, int64_t o_ld, float* S_T,
                              void* saved_states, const void* z, int64_t z_ld,
                              const float* gamma, float eps, void* y, int64_t y_ld,
                              void* workspace, size_t workspace_bytes, uint32_t flags,
                              void* stream) {
  if (!y) return GDN_ERR_INVALID_ARG;
  FwdNorm nm;
  nm.z = z;
  nm.z_ld = z_ld;
  nm.gamma = gamma;
  nm.eps = eps;
  nm.y = y;
  nm.y_ld = y_ld;
  return forward_impl(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                      dt_bias, cu_seqlens, chunk_offsets, S0, o, o_ld, S_T, saved_states,
                      workspace, workspace_bytes, flags, nm, stream);
}

int gdn_backward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k, int64_t k_ld,
                 const void* v, int64_t v_ld, const float* alpha, int64_t alpha_ld,
                 const float* beta_raw, int64_t beta_ld, const float* a_log,
                 const float* dt_bias, const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                 const float* S0, const void* dO, int64_t dO_ld, const float* dS_T,
                 const void* saved_states, void* dq, int64_t dq_ld, void* dk, int64_t dk_ld,
                 void* dv, int64_t dv_ld, float* dalpha, int64_t dalpha_ld, float* dbeta_raw,
                 int64_t dbeta_ld, float* da_log, float* ddt_bias, float* dS0, void* workspace,
                 size_t workspace_bytes, uint32_t flags, void* stream) {
  GDN_TRY(check_shape(s));
  if (flags & ~(uint32_t)(GDN_FLAG_REUSE_FORWARD | GDN_FLAG_BF16_SAVED_STATES))
    return GDN_ERR_INVALID_ARG;
  int bf16_states = 0;
  GDN_TRY(check_bf16_states(s, flags, &bf16_states));
  GDN_TRY(check_inputs(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                       dt_bias, cu_seqlens, chunk_offsets, S0));
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int64_t T = s->total_tokens;
  GDN_TRY(check_matrix(dO, dO_ld, (int64_t)s->Hv * s->Dv, es, T));
  GDN_TRY(check_vec(dS_T, false));
  GDN_TRY(check_vec(saved_states, s->total_chunks > 0));
  GDN_TRY(check_matrix(dq, dq_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(dk, dk_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(dv, dv_ld, (int64_t)s->Hv * s->Dv, es, T));
  GDN_TRY(check_gate_matrix(dalpha, dalpha_ld, s->Hv, T));
  GDN_TRY(check_gate_matrix(dbeta_raw, dbeta_ld, s->Hv, T));
  GDN_TRY(check_head_vec(da_log));
  GDN_TRY(check_head_vec(ddt_bias));
  GDN_TRY(check_vec(dS0, false));
  GDN_TRY(check_workspace(s, workspace, workspace_bytes, true));
  cudaStream_t st = (cudaStream_t)stream;
  Params p;
  fill_common(p, s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
              dt_bias, cu_seqlens, chunk_offsets, S0, workspace, true);
  p.saved_in = (const float*)saved_states;
  p.dO = dO;
  p.dO_ld = dO_ld;
  p.dS_T = dS_T;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dq_ld = dq_ld;
  p.dk_ld = dk_ld;
  p.dv_ld = dv_ld;
  p.dalpha = dalpha;
  p.dbeta = dbeta_raw;
  p.dalpha_ld = dalpha_ld;
  p.dbeta_ld = dbeta_ld;
  p.da_log = da_log;
  p.ddt_bias = ddt_bias;
  p.dS0 = dS0;
  // with no chunk there is nothing to reuse: the flag is then a no-op
  p.reuse = (flags & GDN_FLAG_REUSE_FORWARD) != 0 && s->total_chunks > 0 ? 1 : 0;
  p.bf16_states = bf16_states;
  p.tag = keep_tag(s, bf16_states);
  (void)cudaGetLastError();  // report only errors of this call's own launches
  g_last_error[0] = 0;
  // status block and the fused backward's flags; a reusing backward keeps the
  // forward's tag (it sits after the status word) and clears the flags on their own
  const gdn::WsLayout L = gdn::ws_layout(*s, true);
  cudaError_t e = p.reuse ? cudaMemsetAsync(workspace, 0, sizeof(int32_t) * 2, st)
                          : cudaMemsetAsync(workspace, 0, L.nq, st);
  if (e == cudaSuccess && p.reuse)
    e = cudaMemsetAsync((uint8_t*)workspace + L.bsync, 0, L.nq - L.bsync, st);
  if (e != cudaSuccess) return cuda_fail("gdn_backward: clearing the status word", e);
  if (s->total_chunks == 0 && s->n_seqs > 0 && dS0) {
    const size_t bytes = (size_t)s->n_seqs * s->Hv * s->Dk * s->Dv * sizeof(float);
    e = dS_T ? cudaMemcpyAsync(dS0, dS_T, bytes, cudaMemcpyDeviceToDevice, st)
             : cudaMemsetAsync(dS0, 0, bytes, st);
    if (e != cudaSuccess) return cuda_fail("gdn_backward: dS_0 of empty sequences", e);
  }
  gdn::TmaMaps maps;
  const bool bf16 = s->dtype == GDN_DTYPE_BF16;
  if (bf16 && s->total_tokens > 0) {
    const int64_t T = s->total_tokens;
    if (!gdn::encode_tma_2d(&maps.q, q, (int64_t)s->Hk * s->Dk, T, q_ld) ||
        !gdn::encode_tma_2d(&maps.k, k, (int64_t)s->Hk * s->Dk, T, k_ld) ||
        !gdn::encode_tma_2d(&maps.v, v, (int64_t)s->Hv * s->Dv, T, v_ld) ||
        !gdn::encode_tma_2d(&maps.dO, dO, (int64_t)s->Hv * s->Dv, T, dO_ld)) {
      snprintf(g_last_error, sizeof(g_last_error), "gdn_backward: cuTensorMapEncodeTiled failed");
      return GDN_ERR_CUDA;
    }
  }
  e = gdn::launch_backward(p, bf16 ? &maps : nullptr, st);
  if (e != cudaSuccess) return cuda_fail("gdn_backward: kernel launch", e);
  return GDN_OK;
}

int gdn_decode_step(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                    int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                    int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                    const float* a_log, const float* dt_bias, const float* S_in, float* S_out,
                    void* o, int64_t o_ld, void* stream) {
  if (!s) return GDN_ERR_INVALID_ARG;
  // one token per sequence: the token and chunk counts are the sequence count
  gdn_shape one = *s;
  one.total_tokens = s->n_seqs;
  one.total_chunks = s->n_seqs;
  GDN_TRY(check_shape(&one));
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int64_t N = s->n_seqs;
  GDN_TRY(check_matrix(q, q_ld, (int64_t)s->Hk * s->Dk, es, N));
  GDN_TRY(check_matrix(k, k_ld, (int64_t)s->Hk * s->Dk, es, N));
  GDN_TRY(check_matrix(v, v_ld, (int64_t)s->Hv * s->Dv, es, N));
  GDN_TRY(check_matrix(o, o_ld, (int64_t)s->Hv * s->Dv, es, N));
  GDN_TRY(check_gate_matrix(alpha, alpha_ld, s->Hv, N));
  GDN_TRY(check_gate_matrix(beta_raw, beta_ld, s->Hv, N));
  GDN_TRY(check_head_vec(a_log));
  GDN_TRY(check_head_vec(dt_bias));
  GDN_TRY(check_vec(S_in, false));
  GDN_TRY(check_vec(S_out, N > 0));
  if (N == 0) return GDN_OK;
  (void)cudaGetLastError();  // report only errors of this call's own launch
  g_last_error[0] = 0;
  const cudaError_t e = gdn::launch_decode(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld,
                                           beta_raw, beta_ld, a_log, dt_bias, S_in, S_out, o,
                                           o_ld, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_decode_step: kernel launch", e);
  return GDN_OK;
}

size_t gdn_conv1d_silu_workspace_bytes(int64_t total_tokens, int32_t channels,
                                       int32_t kernel_size) {
  if (total_tokens <= 0 || channels <= 0 || kernel_size <= 0) return 0;
  return gdn::align256(gdn::conv_partial_floats(total_tokens, channels, kernel_size) * 4);
}

size_t gdn_gated_rmsnorm_workspace_bytes(int32_t head_dim) {
  if (head_dim <= 0) return 0;
  return gdn::align256(gdn::norm_partial_floats(head_dim) * 4);
}

int gdn_conv1d_silu_forward(int32_t dtype, int64_t total_tokens, int32_t channels,
                            int32_t kernel_size, const int32_t* cu_seqlens, int32_t n_seqs,
                            const void* x, int64_t x_ld, const float* w, void* y, int64_t y_ld,
                            void* stream) {
  size_t es = 0;
  const int64_t T = total_tokens;
  GDN_TRY(check_conv(dtype, T, channels, kernel_size, cu_seqlens, n_seqs, w, &es));
  GDN_TRY(check_matrix(x, x_ld, channels, es, T));
  GDN_TRY(check_matrix(y, y_ld, channels, es, T));
  if (overlaps(x, x_ld, y, y_ld, T, channels, es)) return GDN_ERR_INVALID_ARG;
  if (T == 0) return GDN_OK;
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  const cudaError_t e = gdn::launch_conv1d_silu(
      false, dtype, T, channels, kernel_size, cu_seqlens, n_seqs, x, x_ld, w, nullptr, 0, y, y_ld,
      nullptr, nullptr, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_conv1d_silu_forward: kernel launch", e);
  return GDN_OK;
}

int gdn_conv1d_silu_backward(int32_t dtype, int64_t total_tokens, int32_t channels,
                             int32_t kernel_size, const int32_t* cu_seqlens, int32_t n_seqs,
                             const void* x, int64_t x_ld, const float* w, const void* dy,
                             int64_t dy_ld, void* dx, int64_t dx_ld, float* dw, void* workspace,
                             size_t workspace_bytes, void* stream) {
  size_t es = 0;
  const int64_t T = total_tokens;
  GDN_TRY(check_conv(dtype, T, channels, kernel_size, cu_seqlens, n_seqs, w, &es));
  GDN_TRY(check_matrix(x, x_ld, channels, es, T));
  GDN_TRY(check_matrix(dy, dy_ld, channels, es, T));
  GDN_TRY(check_matrix(dx, dx_ld, channels, es, T));
  GDN_TRY(check_vec(dw, false));
  if (overlaps(x, x_ld, dx, dx_ld, T, channels, es) ||
      overlaps(dy, dy_ld, dx, dx_ld, T, channels, es))
    return GDN_ERR_INVALID_ARG;
  if (dw)
    GDN_TRY(check_scratch(workspace, workspace_bytes,
                          gdn_conv1d_silu_workspace_bytes(T, channels, kernel_size)));
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  cudaError_t e = cudaSuccess;
  if (T == 0) {
    if (dw) e = cudaMemsetAsync(dw, 0, sizeof(float) * channels * kernel_size, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail("gdn_conv1d_silu_backward: cudaMemsetAsync", e);
    return GDN_OK;
  }
  e = gdn::launch_conv1d_silu(true, dtype, T, channels, kernel_size, cu_seqlens, n_seqs, x, x_ld,
                              w, dy, dy_ld, dx, dx_ld, dw, (float*)workspace,
                              (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_conv1d_silu_backward: kernel launch", e);
  return GDN_OK;
}

int gdn_gated_rmsnorm_forward(int32_t dtype, int64_t total_tokens, int32_t n_heads,
                              int32_t head_dim, float eps, const void* o, int64_t o_ld,
                              const void* z, int64_t z_ld, const float* gamma, void* y,
                              int64_t y_ld, void* stream) {
  size_t es = 0;
  const int64_t T = total_tokens, W = (int64_t)n_heads * head_dim;
  GDN_TRY(check_norm(dtype, T, n_heads, head_dim, eps, gamma, &es));
  GDN_TRY(check_matrix(o, o_ld, W, es, T));
  GDN_TRY(check_matrix(z, z_ld, W, es, T));
  GDN_TRY(check_matrix(y, y_ld, W, es, T));
  if (overlaps(o, o_ld, y, y_ld, T, W, es) || overlaps(z, z_ld, y, y_ld, T, W, es))
    return GDN_ERR_INVALID_ARG;
  if (T == 0) return GDN_OK;
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  const cudaError_t e = gdn::launch_gated_rmsnorm(
      false, dtype, T, n_heads, head_dim, eps, o, o_ld, z, z_ld, gamma, nullptr, 0, y, y_ld,
      nullptr, 0, nullptr, nullptr, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_gated_rmsnorm_forward: kernel launch", e);
  return GDN_OK;
}

int gdn_gated_rmsnorm_backward(int32_t dtype, int64_t total_tokens, int32_t n_heads,
                               int32_t head_dim, float eps, const void* o, int64_t o_ld,
                               const void* z, int64_t z_ld, const float* gamma, const void* dy,
                               int64_t dy_ld, void* d_o, int64_t do_ld, void* dz, int64_t dz_ld,
                               float* dgamma, void* workspace, size_t workspace_bytes,
                               void* stream) {
  size_t es = 0;
  const int64_t T = total_tokens, W = (int64_t)n_heads * head_dim;
  GDN_TRY(check_norm(dtype, T, n_heads, head_dim, eps, gamma, &es));
  GDN_TRY(check_matrix(o, o_ld, W, es, T));
  GDN_TRY(check_matrix(z, z_ld, W, es, T));
  GDN_TRY(check_matrix(dy, dy_ld, W, es, T));
  GDN_TRY(check_matrix(d_o, do_ld, W, es, T));
  GDN_TRY(check_matrix(dz, dz_ld, W, es, T));
  GDN_TRY(check_vec(dgamma, false));
  const void* ins[3] = {o, z, dy};
  const int64_t lds[3] = {o_ld, z_ld, dy_ld};
  for (int i = 0; i < 3; ++i)
    if (overlaps(ins[i], lds[i], d_o, do_ld, T, W, es) || overlaps(ins[i], lds[i], dz, dz_ld, T, W, es))
      return GDN_ERR_INVALID_ARG;
  if (overlaps(d_o, do_ld, dz, dz_ld, T, W, es)) return GDN_ERR_INVALID_ARG;
  if (dgamma)
    GDN_TRY(check_scratch(workspace, workspace_bytes, gdn_gated_rmsnorm_workspace_bytes(head_dim)));
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  cudaError_t e = cudaSuccess;
  if (T == 0) {
    if (dgamma) e = cudaMemsetAsync(dgamma, 0, sizeof(float) * head_dim, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail("gdn_gated_rmsnorm_backward: cudaMemsetAsync", e);
    return GDN_OK;
  }
  e = gdn::launch_gated_rmsnorm(true, dtype, T, n_heads, head_dim, eps, o, o_ld, z, z_ld, gamma,
                                dy, dy_ld, d_o, do_ld, dz, dz_ld, dgamma, (float*)workspace,
                                (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_gated_rmsnorm_backward: kernel launch", e);
  return GDN_OK;
}

int gdn_state_compose(int32_t n, int32_t Dk, int32_t Dv, const float* Phi, const float* S,
                      const float* R, float* out, int32_t transpose, void* stream) {
  if (n < 0 || Dk <= 0 || Dv <= 0 || Dk > 4096 || Dv > 4096 || (transpose != 0 && transpose != 1))
    return GDN_ERR_INVALID_ARG;
  if (n > 65535) return GDN_ERR_UNSUPPORTED;
  GDN_TRY(check_vec(Phi, n > 0));
  GDN_TRY(check_vec(S, n > 0));
  GDN_TRY(check_vec(R, false));
  GDN_TRY(check_vec(out, n > 0));
  const int64_t sz = (int64_t)n * Dk * Dv;
  if (overlaps(Phi, 0, out, 0, 1, (int64_t)n * Dk * Dk, 4) || overlaps(S, 0, out, 0, 1, sz, 4))
    return GDN_ERR_INVALID_ARG;
  if (R && R != out && overlaps(R, 0, out, 0, 1, sz, 4)) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  const cudaError_t e = gdn::launch_state_compose(n, Dk, Dv, Phi, S, R, out, transpose != 0,
                                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_state_compose: kernel launch", e);
  return GDN_OK;
}

int gdn_kda_forward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                    int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                    int64_t alpha_ld, const float* beta_raw, int64_t beta_ld, const float* a_log,
                    const float* b_alpha, const int32_t* cu_seqlens, const float* S_in,
                    float* S_out, void* o, int64_t o_ld, void* stream) {
  if (!s) return GDN_ERR_INVALID_ARG;
  gdn_shape sh = *s;
  // chunks are not used (no saved states); a count consistent with total_tokens
  sh.total_chunks = (int32_t)((s->total_tokens + gdn::kChunk - 1) / gdn::kChunk);
  GDN_TRY(check_shape(&sh));
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int64_t T = s->total_tokens;
  if (T > ((int64_t)1 << 31) - 1) return GDN_ERR_UNSUPPORTED;
  GDN_TRY(check_matrix(q, q_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(k, k_ld, (int64_t)s->Hk * s->Dk, es, T));
  GDN_TRY(check_matrix(v, v_ld, (int64_t)s->Hv * s->Dv, es, T));
  GDN_TRY(check_matrix(o, o_ld, (int64_t)s->Hv * s->Dv, es, T));
  GDN_TRY(check_gate_matrix(alpha, alpha_ld, (int64_t)s->Hv * s->Dk, T));
  GDN_TRY(check_gate_matrix(beta_raw, beta_ld, s->Hv, T));
  GDN_TRY(check_vec(a_log, true));
  GDN_TRY(check_vec(b_alpha, true));
  GDN_TRY(check_vec(S_in, false));
  GDN_TRY(check_vec(S_out, s->n_seqs > 0));
  if (s->n_seqs > 0 && (!cu_seqlens || ((uintptr_t)cu_seqlens & 3u) != 0))
    return cu_seqlens ? GDN_ERR_MISALIGNED : GDN_ERR_INVALID_ARG;
  if (s->n_seqs == 0) return GDN_OK;
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  const cudaError_t e = gdn::launch_kda_forward(&sh, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld,
                                                beta_raw, beta_ld, a_log, b_alpha, cu_seqlens,
                                                S_in, S_out, o, o_ld, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_kda_forward: kernel launch", e);
  return GDN_OK;
}

// Workspace of the chunked KDA forward: status block and work counters, then per (chunk,
// value head) the preparation's tiles (W, K e^{G_last - G}, Q e^G, U^T, P), e^{G_last}
// and the walk's S^T and Delta^T tiles for the output pass.
struct KdaChunkedLayout {
  size_t status, sync, Wsw, Kcw, Qgw, Utb, Psw, Gl, Stb, Dtb, total;
};
static KdaChunkedLayout kda_chunked_layout(const gdn_shape& s) {
  KdaChunkedLayout L{};
  const size_t NCH = (size_t)s.total_chunks * s.Hv, C = gdn::kChunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = gdn::align256(off + bytes);
    return at;
  };
  L.status = take(256);
  L.sync = take(256);
  L.Wsw = take(NCH * gdn::tile_CxD(s.Dk));
  L.Kcw = take(NCH * gdn::tile_CxD(s.Dk));
  L.Qgw = take(NCH * gdn::tile_CxD(s.Dk));
  L.Utb = take(NCH * (size_t)s.Dv * C * 2);
  L.Psw = take(NCH * 8192);
  L.Gl = take(NCH * (size_t)s.Dk * 4);
  L.Stb = take(NCH * gdn::state_tile_bytes(s.Dk, s.Dv));
  L.Dtb = take(NCH * (size_t)s.Dv * 128);
  L.total = off;
  return L;
}

static bool kda_chunked_shape_ok(const gdn_shape* s) {
  return s->dtype == GDN_DTYPE_BF16 && (s->Dk == 64 || s->Dk == 128) &&
         (s->Dv == 64 || s->Dv == 128);
}

size_t gdn_kda_forward_chunked_workspace_bytes(const gdn_shape* s) {
  if (!s || check_shape(s) != GDN_OK || !kda_chunked_shape_ok(s)) return 0;
  return kda_chunked_layout(*s).total;
}

int gdn_kda_forward_chunked(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                            int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                            int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                            const float* a_log, const float* b_alpha,
                            const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                            const float* S_in, float* S_out, void* o, int64_t o_ld,
                            void* workspace, size_t workspace_bytes, void* stream) {
  GDN_TRY(check_shape(s));
  if (!kda_chunked_shape_ok(s)) return GDN_ERR_UNSUPPORTED;
  const int64_t T = s->total_tokens;
  if (T > ((int64_t)1 << 31) - 1) return GDN_ERR_UNSUPPORTED;
  GDN_TRY(check_matrix(q, q_ld, (int64_t)s->Hk * s->Dk, 2, T));
  GDN_TRY(check_matrix(k, k_ld, (int64_t)s->Hk * s->Dk, 2, T));
  GDN_TRY(check_matrix(v, v_ld, (int64_t)s->Hv * s->Dv, 2, T));
  GDN_TRY(check_matrix(o, o_ld, (int64_t)s->Hv * s->Dv, 2, T));
  GDN_TRY(check_gate_matrix(alpha, alpha_ld, (int64_t)s->Hv * s->Dk, T));
  GDN_TRY(check_gate_matrix(beta_raw, beta_ld, s->Hv, T));
  GDN_TRY(check_vec(a_log, true));
  GDN_TRY(check_vec(b_alpha, true));
  GDN_TRY(check_vec(S_in, false));
  GDN_TRY(check_vec(S_out, s->n_seqs > 0));
  if (s->n_seqs > 0) {
    if (!cu_seqlens || !chunk_offsets) return GDN_ERR_INVALID_ARG;
    if (((uintptr_t)cu_seqlens & 3u) != 0 || ((uintptr_t)chunk_offsets & 3u) != 0)
      return GDN_ERR_MISALIGNED;
  }
  const KdaChunkedLayout L = kda_chunked_layout(*s);
  if (!workspace || ((uintptr_t)workspace & 255u) != 0 || workspace_bytes < L.total)
    return GDN_ERR_WORKSPACE;
  if (s->n_seqs == 0) return GDN_OK;
  cudaStream_t st = (cudaStream_t)stream;
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  cudaError_t e = cudaMemsetAsync(workspace, 0, L.Wsw, st);   // status and counters
  if (e != cudaSuccess) return cuda_fail("gdn_kda_forward_chunked: clearing the status word", e);
  if (s->total_chunks == 0) {   // every sequence is empty: S_out = S_in
    const size_t bytes = (size_t)s->n_seqs * s->Hv * s->Dk * s->Dv * sizeof(float);
    e = S_in ? (S_in == S_out ? cudaSuccess
                              : cudaMemcpyAsync(S_out, S_in, bytes, cudaMemcpyDeviceToDevice, st))
             : cudaMemsetAsync(S_out, 0, bytes, st);
    return e == cudaSuccess ? GDN_OK : cuda_fail("gdn_kda_forward_chunked: empty sequences", e);
  }
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.Hk = s->Hk;
  p.Hv = s->Hv;
  p.Dk = s->Dk;
  p.Dv = s->Dv;
  p.r = s->Hv / s->Hk;
  p.head_map = s->head_map;
  p.n_seqs = s->n_seqs;
  p.NC = s->total_chunks;
  p.T = T;
  p.scale = s->scale > 0.f ? s->scale : 1.0f / std::sqrt((float)s->Dk);
  p.q = q;
  p.k = k;
  p.v = v;
  p.q_ld = q_ld;
  p.k_ld = k_ld;
  p.v_ld = v_ld;
  p.alpha = alpha;
  p.alpha_ld = alpha_ld;
  p.beta_raw = beta_raw;
  p.beta_ld = beta_ld;
  p.a_log = a_log;
  p.b_alpha = b_alpha;
  p.cu = cu_seqlens;
  p.coff = chunk_offsets;
  p.S0 = S_in;
  p.S_T = S_out;
  p.o = o;
  p.o_ld = o_ld;
  p.kda = 1;
  char* base = (char*)workspace;
  p.status = (gdn::DeviceStatus*)(base + L.status);
  p.fwork = (uint32_t*)(base + L.sync);
  p.Wsw = (uint8_t*)(base + L.Wsw);
  p.Kcw = (uint8_t*)(base + L.Kcw);
  p.Qgw = (uint8_t*)(base + L.Qgw);
  p.Utb = (__nv_bfloat16*)(base + L.Utb);
  p.Psw = (uint8_t*)(base + L.Psw);
  p.Gl = (float*)(base + L.Gl);
  p.Stb = (uint8_t*)(base + L.Stb);
  p.Dtb = (uint8_t*)(base + L.Dtb);
  gdn::TmaMaps maps;
  if (!gdn::encode_tma_2d(&maps.q, q, (int64_t)s->Hk * s->Dk, T, q_ld) ||
      !gdn::encode_tma_2d(&maps.k, k, (int64_t)s->Hk * s->Dk, T, k_ld) ||
      !gdn::encode_tma_2d(&maps.v, v, (int64_t)s->Hv * s->Dv, T, v_ld)) {
    snprintf(g_last_error, sizeof(g_last_error),
             "gdn_kda_forward_chunked: cuTensorMapEncodeTiled failed");
    return GDN_ERR_CUDA;
  }
  e = gdn::launch_kda_prep_tc(p, maps, st);
  if (e == cudaSuccess) e = gdn::launch_fwd_state_tc(p, st);
  if (e == cudaSuccess) e = gdn::launch_fwd_out_tc(p, st);
  if (e != cudaSuccess) return cuda_fail("gdn_kda_forward_chunked: kernel launch", e);
  return GDN_OK;
}

size_t gdn_kda_backward_workspace_bytes(const gdn_shape* s) {
  if (!s || s->total_tokens < 0 || s->n_seqs < 0 || s->Hv <= 0 || s->Dk <= 0 || s->Dv <= 0)
    return 0;
  return gdn::align256(gdn::kda_bwd_workspace_floats(s) * sizeof(float));
}

int gdn_kda_backward(const gdn_shape* s, const void* q, int64_t q_ld, const void* k,
                     int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                     int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                     const float* a_log, const float* b_alpha, const int32_t* cu_seqlens,
                     const float* S0, const void* dO, int64_t dO_ld, const float* dS_T,
                     void* dq, int64_t dq_ld, void* dk, int64_t dk_ld, void* dv, int64_t dv_ld,
                     float* dalpha, int64_t dalpha_ld, float* dbeta_raw, int64_t dbeta_ld,
                     float* da_log, float* db_alpha, float* dS0, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!s) return GDN_ERR_INVALID_ARG;
  gdn_shape sh = *s;
  sh.total_chunks = (int32_t)((s->total_tokens + gdn::kChunk - 1) / gdn::kChunk);
  GDN_TRY(check_shape(&sh));
  if (s->Dv < 32) return GDN_ERR_UNSUPPORTED;  // 32-column slices
  const size_t es = s->dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int64_t T = s->total_tokens;
  if (T > ((int64_t)1 << 31) - 1 || s->n_seqs > 65535) return GDN_ERR_UNSUPPORTED;
  const int64_t wk = (int64_t)s->Hk * s->Dk, wv = (int64_t)s->Hv * s->Dv;
  GDN_TRY(check_matrix(q, q_ld, wk, es, T));
  GDN_TRY(check_matrix(k, k_ld, wk, es, T));
  GDN_TRY(check_matrix(v, v_ld, wv, es, T));
  GDN_TRY(check_matrix(dO, dO_ld, wv, es, T));
  GDN_TRY(check_matrix(dq, dq_ld, wk, es, T));
  GDN_TRY(check_matrix(dk, dk_ld, wk, es, T));
  GDN_TRY(check_matrix(dv, dv_ld, wv, es, T));
  GDN_TRY(check_gate_matrix(alpha, alpha_ld, (int64_t)s->Hv * s->Dk, T));
  GDN_TRY(check_gate_matrix(dalpha, dalpha_ld, (int64_t)s->Hv * s->Dk, T));
  GDN_TRY(check_gate_matrix(beta_raw, beta_ld, s->Hv, T));
  GDN_TRY(check_gate_matrix(dbeta_raw, dbeta_ld, s->Hv, T));
  GDN_TRY(check_vec(a_log, true));
  GDN_TRY(check_vec(b_alpha, true));
  GDN_TRY(check_vec(da_log, true));
  GDN_TRY(check_vec(db_alpha, true));
  GDN_TRY(check_vec(S0, false));
  GDN_TRY(check_vec(dS_T, false));
  GDN_TRY(check_vec(dS0, false));
  if (s->n_seqs > 0 && (!cu_seqlens || ((uintptr_t)cu_seqlens & 3u) != 0))
    return cu_seqlens ? GDN_ERR_MISALIGNED : GDN_ERR_INVALID_ARG;
  GDN_TRY(check_scratch(workspace, workspace_bytes, gdn_kda_backward_workspace_bytes(s)));
  (void)cudaGetLastError();
  g_last_error[0] = 0;
  cudaError_t e = cudaSuccess;
  if (s->n_seqs == 0) {  // nothing to walk: the parameter gradients are zero
    e = cudaMemsetAsync(da_log, 0, sizeof(float) * s->Hv, (cudaStream_t)stream);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(db_alpha, 0, sizeof(float) * s->Hv * s->Dk, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail("gdn_kda_backward: cudaMemsetAsync", e);
    return GDN_OK;
  }
  e = gdn::launch_kda_backward(&sh, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld,
                               a_log, b_alpha, cu_seqlens, S0, dO, dO_ld, dS_T, dq, dq_ld, dk,
                               dk_ld, dv, dv_ld, dalpha, dalpha_ld, dbeta_raw, dbeta_ld, da_log,
                               db_alpha, dS0, (float*)workspace, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("gdn_kda_backward: kernel launch", e);
  return GDN_OK;
}

int gdn_read_device_status(const void* workspace, void* stream) {
  if (!workspace) return GDN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  gdn::DeviceStatus h{};
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail("gdn_read_device_status: copy", e);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail("gdn_read_device_status: synchronize", e);
  return h.code;
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_DEVICE_BOUNDS: return "GDN_ERR_DEVICE_BOUNDS";
    case GDN_ERR_NOT_KEPT: return "GDN_ERR_NOT_KEPT";
    default: return "GDN_UNKNOWN_STATUS";
  }
}

}  // extern "C"
