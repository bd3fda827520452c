/*
 * gdn.h -- C ABI of the GB300 Gated DeltaNet library (libgdn.so).
 *
 * The operation (lattice-inference 0.6.0, src/attention/gdn_backward.rs,
 * module doc "Forward recap"): for every sequence of a varlen batch and every
 * value head h, with key head kh = h / (Hv / Hk),
 *
 *   q_hat = q / sqrt(|q|^2 + 1e-6),  k_hat = k / sqrt(|k|^2 + 1e-6)   (key head kh)
 *   beta  = sigmoid(beta_raw[t, h])
 *   g     = exp(-exp(a_log[h]) * softplus(alpha[t, h] + dt_bias[h]))
 *   kv    = S_{t-1}^T k_hat                 (retrieval from the pre-decayed state)
 *   delta = beta * (v - g * kv)
 *   S_t   = g * S_{t-1} + k_hat delta^T     (S is Dk x Dv, row-major)
 *   o_t   = scale * S_t^T q_hat             (scale = 1/sqrt(Dk) unless given)
 *
 * The backward is its reverse-mode derivative (gdn_backward, section 4,
 * steps 4a-4h), taking dO and dS_T and returning dq, dk, dv, d alpha,
 * d beta_raw, d a_log, d dt_bias and dS_0.  dq/dk of a key head are the sums
 * over the value heads that read it (the cross-head reduction of the llama.cpp
 * PR "tests: delta-net backward at the shape the 27B emits (shared key heads,
 * strided q/k)"), formed in a fixed order: results are bit-reproducible run to
 * run.  q/k/v may be strided row views of one packed projection (same PR).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Tokens of all sequences are packed row after row; sequence n owns rows
 *    [cu_seqlens[n], cu_seqlens[n+1]).  Each sequence starts from its own S_0.
 *  - `*_ld` arguments are row strides in ELEMENTS (one row per token).  Inside a
 *    row, head h occupies columns [h*D, (h+1)*D).
 *  - q, k, v, o, dO, dq, dk, dv have the element type `shape->dtype` (fp32 or
 *    bf16).  alpha, beta_raw, a_log, dt_bias, S_0, S_T, dS_T, dS_0 and d alpha,
 *    d beta_raw, d a_log, d dt_bias are fp32.  State and accumulation
 *    arithmetic is fp32.  bf16 outputs are rounded to nearest even.
 *  - State tensors (S_0, S_T, dS_T, dS_0) are [n_seqs, Hv, Dk, Dv] fp32,
 *    contiguous.
 *  - Saved states hold the state at the START of each 64-token chunk (chunks
 *    never span two sequences; the last chunk of a sequence may be short; the
 *    chunks of sequence n are numbered from chunk_offsets[n]), one block per
 *    (chunk, value head), chunk-major.  fp32 inputs: [total_chunks, Hv, Dk, Dv]
 *    fp32.  bf16 inputs: the state is kept in bf16, as the operand tile of the
 *    backward's tensor-core products, S^T with MV = max(Dv, 64) rows (v) and
 *    Dk columns (k), 128-byte-swizzled K-major: element (v, k) is the bf16 at
 *    byte ((k / 64) * MV + v) * 128 + ((((k % 64) / 8) ^ (v % 8)) * 16) +
 *    (k % 8) * 2 of its block (padding rows and columns hold zero); a block is
 *    ceil(Dk / 64) * MV * 128 bytes.
 *  - Pointers marked "device" are CUDA device pointers; "host" ones are host
 *    pointers.  The caller owns every buffer.  The library allocates nothing
 *    and keeps no state between calls.  Outputs are overwritten, never
 *    accumulated into.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and the call returns without synchronising.
 *  - Every argument is checked on the host before anything is launched: on a
 *    failed check the call returns a negative gdn_status and launches nothing.
 *    Supported: Dk, Dv in {16, 32, 64, 128}; Hv a multiple of Hk; device
 *    buffers 16-byte aligned, except the fp32 per-head gate matrices alpha,
 *    beta_raw, d alpha, d beta_raw and vectors a_log, dt_bias, d a_log,
 *    d dt_bias, which need 4-byte alignment (so that a column slice of them, one
 *    rank's heads, can be passed as it is); row strides of q, k, v, o, dO, dq,
 *    dk, dv whose byte size is a multiple of 16; fp32 row strides of alpha,
 *    beta_raw, d alpha, d beta_raw of at least Hv; workspace at least
 *    gdn_workspace_bytes() and 256-byte aligned.
 *  - Errors found on the device (a cu_seqlens / chunk_offsets pair that does
 *    not match the shape, a bounded wait that ran out) do not trap: the kernels
 *    record a status code in the workspace and skip the offending work.  Read it
 *    with gdn_read_device_status().
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1,   /* null pointer, bad size, inconsistent cu_seqlens */
  GDN_ERR_UNSUPPORTED = -2,   /* head size or dtype outside the supported set */
  GDN_ERR_MISALIGNED = -3,    /* pointer or row stride breaks the alignment rules */
  GDN_ERR_CUDA = -4,          /* a CUDA runtime call or a launch failed */
  GDN_ERR_TIMEOUT = -5,       /* a bounded device-side wait ran out (device status) */
  GDN_ERR_WORKSPACE = -6,     /* workspace too small or misaligned */
  GDN_ERR_DEVICE_BOUNDS = -7, /* device-side check: chunk or token index out of range */
  GDN_ERR_NOT_KEPT = -8       /* GDN_FLAG_REUSE_FORWARD given a workspace that holds no
                                 kept forward of this shape (device status) */
} gdn_status;

typedef enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

/* Call flags (the `flags` argument of gdn_forward / gdn_backward).
 *
 * A training step runs the forward and then, on the same inputs, the backward.
 * Both need the same per-chunk operands (normalised q/k tiles, the gates, the
 * inverse T = (I + A)^-1 and W, U, P of each chunk and value head).  With
 * GDN_FLAG_KEEP_FOR_BACKWARD the forward leaves them in its workspace, which
 * must then be gdn_workspace_bytes(shape, 1) bytes, and stamps the workspace
 * with a tag of the shape.  The backward, given that same workspace untouched
 * in between and GDN_FLAG_REUSE_FORWARD, reads them instead of recomputing
 * them.  Results are bit-identical to a backward without the flag.  A REUSE
 * backward whose workspace carries no matching tag computes nothing and
 * records GDN_ERR_NOT_KEPT as its device status; the host cannot see the tag
 * without synchronising, so the call itself returns GDN_OK.  Keeping the
 * operands for inputs that then change before the backward is the caller's
 * error and is not detected. */
typedef enum {
  GDN_FLAG_KEEP_FOR_BACKWARD = 1, /* gdn_forward only */
  GDN_FLAG_REUSE_FORWARD = 2,     /* gdn_backward only */
  GDN_FLAG_BF16_SAVED_STATES = 4  /* gdn_forward and gdn_backward; see below */
} gdn_flag;

/* GDN_FLAG_BF16_SAVED_STATES (a measured option of this library; the default is the
 * fp32 layout below).  For bf16 inputs with Dk, Dv >= 64 the forward may keep the
 * chunk-start states in bf16, the precision every tensor-core product that reads them
 * rounds them to anyway, as one tile of S^T per (chunk, value head): max(Dv, 64) rows
 * (value index) by Dk columns (key index), each 64-column block stored as 128-byte rows
 * whose 16-byte pieces are XOR-permuted by row % 8 (the K-major 128-byte-swizzled
 * operand layout of the tensor cores): element (v, k) at byte
 *   (k / 64) * max(Dv, 64) * 128 + v * 128 + (((k % 64) / 8) ^ (v % 8)) * 16 + (k % 8) * 2
 * of the tile, tiles ceil(Dk / 64) * max(Dv, 64) * 128 bytes apart in (chunk, value
 * head) order.  That halves the largest byte stream of a training step; the gradients
 * are the same bits as with fp32 states (the backward rounds the fp32 states to the
 * same bf16 values).  The backward must be given the same flag as the forward that
 * wrote the buffer.  With fp32 inputs or a head size below 64 the flag returns
 * GDN_ERR_UNSUPPORTED. */

/* Key head of value head h (v_repeat = Hv / Hk value heads share each key head).
 * GDN_HEAD_MAP_CONSECUTIVE: kh = h / v_repeat (value heads kh*v_repeat ..
 * kh*v_repeat + v_repeat - 1 share key head kh; the default, and the head map of the
 * Rust forward/backward page).  GDN_HEAD_MAP_MODULO: kh = h % Hk (value heads kh,
 * kh + Hk, kh + 2 Hk, ... share key head kh; the broadcast the ggml page's op uses).
 * Every other argument keeps its meaning; dq / dk still sum over the value heads that
 * read the key head. */
typedef enum { GDN_HEAD_MAP_CONSECUTIVE = 0, GDN_HEAD_MAP_MODULO = 1 } gdn_head_map;

typedef struct {
  int32_t Hk;           /* key heads (q and k heads) */
  int32_t Hv;           /* value heads; Hv % Hk == 0, v_repeat = Hv / Hk */
  int32_t Dk;           /* key / query head size */
  int32_t Dv;           /* value head size */
  int32_t n_seqs;       /* sequences in the varlen batch (>= 0) */
  int32_t total_chunks; /* sum over sequences of ceil(len / 64), from gdn_plan */
  int64_t total_tokens; /* cu_seqlens[n_seqs] */
  int32_t dtype;        /* gdn_dtype of q, k, v, o, dO, dq, dk, dv */
  float scale;          /* output scale; 0 selects 1/sqrt(Dk) */
  int32_t head_map;     /* gdn_head_map: which key head value head h reads */
} gdn_shape;

/* Chunk planning (host only).  From host cu_seqlens[n_seqs+1] (non-decreasing,
 * starting at 0) fills chunk_offsets_host[n_seqs+1] (chunk_offsets[n] = number
 * of 64-token chunks of the sequences before n) and *total_chunks.  The caller
 * copies both arrays to the device for gdn_forward / gdn_backward.
 * Returns GDN_OK or GDN_ERR_INVALID_ARG. */
int gdn_plan(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t* chunk_offsets_host,
             int32_t* total_chunks);

/* Bytes of the saved-state buffer: total_chunks * Hv * Dk * Dv * 4.  It holds the
 * state S at the start of every chunk, fp32 [total_chunks, Hv, Dk, Dv] row-major
 * (chunk c of sequence n at index chunk_offsets[n] + c; S[i][j] at i * Dv + j, i over
 * the key index), for both input dtypes; GDN_FLAG_BF16_SAVED_STATES stores bf16 tiles
 * in the first part of the same buffer instead (Dk, Dv >= 64).  Returns 0 for an
 * invalid shape. */
size_t gdn_saved_state_bytes(const gdn_shape* shape);

/* Bytes of device scratch the forward (is_backward = 0) or the backward
 * (is_backward = 1) needs.  Returns 0 for an invalid shape. */
size_t gdn_workspace_bytes(const gdn_shape* shape, int is_backward);

/* Forward.  Chunked (64-token) scan of the recurrence above.
 *   q, k      device, [total_tokens, *_ld] dtype; key head kh at column kh*Dk
 *   v         device, [total_tokens, v_ld] dtype; value head h at column h*Dv
 *   alpha     device, [total_tokens, alpha_ld] fp32; column h
 *   beta_raw  device, [total_tokens, beta_ld] fp32; column h (beta = sigmoid)
 *   a_log, dt_bias  device, [Hv] fp32
 *   cu_seqlens, chunk_offsets  device, [n_seqs+1] int32 (see gdn_plan)
 *   S0        device, [n_seqs, Hv, Dk, Dv] fp32, or NULL for a zero state
 *   o         device, [total_tokens, o_ld] dtype (written)
 *   S_T       device, [n_seqs, Hv, Dk, Dv] fp32 final states, or NULL
 *   saved_states device, gdn_saved_state_bytes() bytes (written: the fp32 state
 *             at the start of every chunk, which the backward reads), or NULL for a
 *             forward no backward will read (prefill, inference: the chunk-start
 *             states are then not stored); required with GDN_FLAG_KEEP_FOR_BACKWARD
 *   workspace device scratch, gdn_workspace_bytes(shape, 0) bytes
 *             (gdn_workspace_bytes(shape, 1) with GDN_FLAG_KEEP_FOR_BACKWARD)
 *   flags     0, or GDN_FLAG_KEEP_FOR_BACKWARD and / or GDN_FLAG_BF16_SAVED_STATES
 * Returns a gdn_status. */
int gdn_forward(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                const float* a_log, const float* dt_bias, const int32_t* cu_seqlens,
                const int32_t* chunk_offsets, const float* S0, void* o, int64_t o_ld,
                float* S_T, void* saved_states, void* workspace, size_t workspace_bytes,
                uint32_t flags, void* stream);

/* Backward (reverse chunk walk with a dS carry).  Inputs as gdn_forward, plus
 *   dO        device, [total_tokens, dO_ld] dtype: dL/do
 *   dS_T      device, [n_seqs, Hv, Dk, Dv] fp32: dL/dS_T, or NULL for zero
 *   saved_states device, as written by gdn_forward on the same inputs (with the
 *             same GDN_FLAG_BF16_SAVED_STATES setting)
 * Outputs (all written, none accumulated):
 *   dq, dk    device, [total_tokens, *_ld] dtype: dL/dq, dL/dk of the RAW
 *             (un-normalised) q and k, summed over the value heads of each key head
 *   dv        device, [total_tokens, dv_ld] dtype
 *   dalpha    device, [total_tokens, dalpha_ld] fp32: dL/d alpha
 *   dbeta_raw device, [total_tokens, dbeta_ld] fp32: dL/d beta_raw
 *   da_log, ddt_bias device, [Hv] fp32, summed over every token of every sequence
 *   dS0       device, [n_seqs, Hv, Dk, Dv] fp32: dL/dS_0, or NULL to skip
 *   workspace device scratch, gdn_workspace_bytes(shape, 1) bytes; with
 *             GDN_FLAG_REUSE_FORWARD, the workspace of the kept forward
 *   flags     0, or GDN_FLAG_REUSE_FORWARD and / or GDN_FLAG_BF16_SAVED_STATES
 * Returns a gdn_status. */
int gdn_backward(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                 int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                 int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                 const float* a_log, const float* dt_bias, const int32_t* cu_seqlens,
                 const int32_t* chunk_offsets, const float* S0, const void* dO, int64_t dO_ld,
                 const float* dS_T, const void* saved_states, void* dq, int64_t dq_ld,
                 void* dk, int64_t dk_ld, void* dv, int64_t dv_ld, float* dalpha,
                 int64_t dalpha_ld, float* dbeta_raw, int64_t dbeta_ld, float* da_log,
                 float* ddt_bias, float* dS0, void* workspace, size_t workspace_bytes,
                 uint32_t flags, void* stream);

/* Size of the scratch array built into the library for gdn_forward_noalloc. */
#define GDN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* gdn_forward for callers that cannot allocate device memory (no counterpart on
 * the pages this library implements; it is a convenience of this library).
 * Some callers may not call cudaMalloc: code that runs under a device-memory
 * budget fixed at start-up, plugin hosts that pass a kernel its inputs and
 * outputs but no scratch, and paths that cannot accept the implicit device
 * synchronisation of cudaMalloc / cudaFree.  This entry point takes the same
 * arguments as gdn_forward minus the workspace and the flags (it keeps nothing
 * for a backward) and uses instead one scratch
 * array of GDN_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library, which
 * every GPU that loads the library holds until the process exits.  It allocates
 * nothing.
 *  - Shapes whose gdn_workspace_bytes(shape, 0) exceeds GDN_NOALLOC_SCRATCH_BYTES
 *    are rejected with GDN_ERR_WORKSPACE before anything is launched
 *    (gdn_last_error() says why); use gdn_forward with a caller workspace.
 *  - The scratch's device address is looked up (cudaGetSymbolAddress, with the
 *    calling device current) on every call made outside stream capture, so a
 *    device reset or another context of the device does not leave a stale
 *    address behind.  A call on a capturing stream reuses the address of that
 *    device's last call outside capture: make the first call on each device
 *    before any stream capture (a first call inside capture returns
 *    GDN_ERR_UNSUPPORTED), and repeat one outside capture after a device reset.
 *  - All calls on a device share the one scratch array, which keeps the last
 *    call's contents (each call clears what must start at zero).  Calls whose
 *    work overlaps on the GPU (concurrent streams, or host threads) race on it:
 *    serialise them.
 *  - The device-side status of these calls is not readable through
 *    gdn_read_device_status (the caller has no workspace pointer).
 * Returns a gdn_status like gdn_forward. */
int gdn_forward_noalloc(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                        int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                        int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                        const float* a_log, const float* dt_bias, const int32_t* cu_seqlens,
                        const int32_t* chunk_offsets, const float* S0, void* o, int64_t o_ld,
                        float* S_T, void* saved_states, void* stream);

/* One decode step: every sequence takes one new token (the recurrence above applied
 * once, in its token form; Gated Delta Networks, the gated delta rule update).  For
 * every sequence n and value head h, with kh = h / (Hv / Hk):
 *   q_hat, k_hat = q / sqrt(|q|^2 + 1e-6), k / sqrt(|k|^2 + 1e-6)   (key head kh)
 *   g = exp(-e^{a_log[h]} softplus(alpha + dt_bias[h])),  beta = sigmoid(beta_raw)
 *   delta = beta (v - g S^T k_hat);  S <- g S + k_hat delta^T;  o = scale S^T q_hat
 * shape: Hk, Hv, Dk, Dv, dtype and scale as for gdn_forward; n_seqs sequences of one
 *   token each (total_tokens and total_chunks are not read).
 *   q, k      device, [n_seqs, *_ld] dtype: the new token's query / key rows
 *   v         device, [n_seqs, v_ld] dtype
 *   alpha, beta_raw  device, [n_seqs, *_ld] fp32
 *   a_log, dt_bias   device, [Hv] fp32
 *   S_in      device, [n_seqs, Hv, Dk, Dv] fp32 state before the token, or NULL
 *             for a zero state
 *   S_out     device, [n_seqs, Hv, Dk, Dv] fp32 state after the token (written);
 *             S_out == S_in updates the state in place; partly overlapping
 *             buffers are not supported
 *   o         device, [n_seqs, o_ld] dtype (written)
 * Needs no workspace and keeps nothing for a backward.  Validation, alignment rules
 * and return values as for gdn_forward (nothing is launched on an error). */
int gdn_decode_step(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                    int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                    int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                    const float* a_log, const float* dt_bias, const float* S_in, float* S_out,
                    void* o, int64_t o_ld, void* stream);

/* ---- The layer steps on either side of the recurrence --------------------------------
 * lattice-inference 0.6.0, src/attention/gdn_backward.rs: the forward's "Causal conv1d +
 * SiLU" step (which makes the recurrence's q|k|v from the packed projection) and "Gated
 * RMSNorm + output projection" step (which normalises o), and their backward (the
 * backward's sections 5 and 2).  They take plain sizes instead of a gdn_shape.  dtype is
 * a gdn_dtype; x, y, dy, dx, o, z and the norm's outputs have that element type, the
 * weights and their gradients are fp32, arithmetic is fp32.  Matrices are [rows, ld] with
 * ld in elements, 16-byte aligned, ld * element size a multiple of 16.  An output may not
 * overlap an input or another output (GDN_ERR_INVALID_ARG).  The weight gradients (dw,
 * d gamma) are optional (NULL skips them); when asked for they are formed in a fixed order
 * from per-block partial sums kept in `workspace` (16-byte aligned, at least the size the
 * matching *_workspace_bytes returns), so they are bit-reproducible run to run.
 *
 * Causal depthwise conv1d + SiLU, channel c of token t of sequence n:
 *   y[t, c] = SiLU(sum_{j<K} w[c*K + j] * x[t - (K-1) + j, c])
 * where inputs before cu_seqlens[n] (the sequence's first token) read as zero: each
 * sequence starts with an empty rolling buffer.  The last tap (j = K-1) is the current
 * token.  Backward, with pre[t, c] the argument of SiLU and d_sum = dy * SiLU'(pre):
 *   dx[s, c] = sum_{j<K} d_sum[s + K-1-j, c] * w[c*K + j]   (terms inside s's sequence)
 *   dw[c*K + j] = sum_t d_sum[t, c] * x[t - (K-1) + j, c]
 *   channels     C, a multiple of 8 (the packed q|k|v width 2 Hk Dk + Hv Dv is one),
 *                at most 2^24;  total_tokens at most 2^30
 *   kernel_size  K in 1..4
 *   cu_seqlens   device, int32 [n_seqs + 1]: 0 = cu[0] <= ... <= cu[n_seqs] = total_tokens
 *                (not checked on the host; a malformed one gives wrong values but every
 *                access stays inside the buffers)
 *   x            device, [total_tokens, x_ld]: the projection rows (q|k|v packed)
 *   w            device, fp32 [C, K]
 *   y            device, [total_tokens, y_ld] (written): q, k and v of gdn_forward are
 *                strided views of it (q = y, k = y + Hk Dk, v = y + 2 Hk Dk, ld = y_ld)
 *   dy           device, [total_tokens, dy_ld]: the gradient of y (dq|dk|dv packed)
 *   dx           device, [total_tokens, dx_ld] (written);  dw  device, fp32 [C, K] or NULL
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_MISALIGNED,
 * GDN_ERR_WORKSPACE or GDN_ERR_CUDA; nothing is launched on an error. */
int gdn_conv1d_silu_forward(int32_t dtype, int64_t total_tokens, int32_t channels,
                            int32_t kernel_size, const int32_t* cu_seqlens, int32_t n_seqs,
                            const void* x, int64_t x_ld, const float* w, void* y, int64_t y_ld,
                            void* stream);
size_t gdn_conv1d_silu_workspace_bytes(int64_t total_tokens, int32_t channels,
                                       int32_t kernel_size);
int gdn_conv1d_silu_backward(int32_t dtype, int64_t total_tokens, int32_t channels,
                             int32_t kernel_size, const int32_t* cu_seqlens, int32_t n_seqs,
                             const void* x, int64_t x_ld, const float* w, const void* dy,
                             int64_t dy_ld, void* dx, int64_t dx_ld, float* dw, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Gated RMSNorm of every (token t, head h) row of head_dim values (o, z of that head):
 *   rms = sqrt(mean_j o_j^2 + eps),   y_j = (o_j / rms) * gamma[j] * SiLU(z_j)
 * with gamma shared by the heads.  Backward, with x_n = o / rms:
 *   d_xn = dy gamma SiLU(z),  dz = dy gamma x_n SiLU'(z),
 *   do = d_xn / rms - o (sum_j d_xn_j o_j) / (rms^3 head_dim),
 *   d gamma[j] = sum over tokens and heads of dy_j x_n,j SiLU(z_j)
 *   n_heads      H >= 1;  head_dim D in {16, 32, 64, 128};  eps >= 0 (finite);
 *                total_tokens * H * D at most 2^31
 *   o, z         device, [total_tokens, *_ld] holding H*D used columns
 *   gamma        device, fp32 [D]
 *   y            device, [total_tokens, y_ld] (written)
 *   dy           device, [total_tokens, dy_ld]: the gradient of y
 *   d_o, dz      device, [total_tokens, *_ld] (written): d_o is the recurrence's dO
 *   dgamma       device, fp32 [D] or NULL
 * Returns as the conv entry points do. */
int gdn_gated_rmsnorm_forward(int32_t dtype, int64_t total_tokens, int32_t n_heads,
                              int32_t head_dim, float eps, const void* o, int64_t o_ld,
                              const void* z, int64_t z_ld, const float* gamma, void* y,
                              int64_t y_ld, void* stream);
size_t gdn_gated_rmsnorm_workspace_bytes(int32_t head_dim);

/* gdn_forward followed by gdn_gated_rmsnorm_forward of its output over the Hv value heads
 * (n_heads = Hv, head_dim = Dv): o as gdn_forward writes it, and y = the gated RMSNorm of
 * each (token, value head) row of o with z, gamma and eps, the norm taken over o as stored
 * (its element type).  With bf16 inputs the norm runs in the epilogue of the forward's
 * output pass, which holds each row's Dv values when it stores them, so y costs one read
 * of z and one write of y instead of a further pass over o; with fp32 inputs it is the
 * separate norm kernel after the forward.  o is still written: the norm's backward reads
 * it.  Arguments as gdn_forward and gdn_gated_rmsnorm_forward:
 *   z, z_ld   device, [total_tokens, z_ld] of the shape's dtype, Hv*Dv used columns
 *   gamma     device, fp32 [Dv];  eps >= 0, finite
 *   y, y_ld   device, [total_tokens, y_ld] of the shape's dtype (written)
 * y must not overlap o or z, and o must not overlap z (GDN_ERR_INVALID_ARG); y NULL is
 * GDN_ERR_INVALID_ARG.  The rows agree with gdn_gated_rmsnorm_forward on this o to within
 * the rounding of the sum of squares (the two sum the row in different orders).
 * Returns a gdn_status. */
int gdn_forward_gated_rmsnorm(const gdn_shape* shape, const void* q, int64_t q_ld,
                              const void* k, int64_t k_ld, const void* v, int64_t v_ld,
                              const float* alpha, int64_t alpha_ld, const float* beta_raw,
                              int64_t beta_ld, const float* a_log, const float* dt_bias,
                              const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                              const float* S0, void* o, int64_t o_ld, float* S_T,
                              void* saved_states, const void* z, int64_t z_ld,
                              const float* gamma, float eps, void* y, int64_t y_ld,
                              void* workspace, size_t workspace_bytes, uint32_t flags,
                              void* stream);
int gdn_gated_rmsnorm_backward(int32_t dtype, int64_t total_tokens, int32_t n_heads,
                               int32_t head_dim, float eps, const void* o, int64_t o_ld,
                               const void* z, int64_t z_ld, const float* gamma, const void* dy,
                               int64_t dy_ld, void* d_o, int64_t do_ld, void* dz, int64_t dz_ld,
                               float* dgamma, void* workspace, size_t workspace_bytes,
                               void* stream);

/* ---- Context parallelism: composing segment state maps ---------------------------------
 * A sequence cut into consecutive segments maps each segment's start state affinely to its
 * end state (the forward recap's update rewritten as S_t = g_t (I - beta_t k_t k_t^T)
 * S_{t-1} + beta_t k_t v_t^T):  S_out = Phi S_in + R, Phi = prod_t g_t (I - beta_t k_t
 * k_t^T) (Dk x Dk, latest token leftmost), R the end state from a zero start; the
 * start-state gradient is dS_in = Phi^T dS_out + G.  Phi is gdn_forward's S_T for the
 * segment run with v = 0 from S_0 = I (a shape with Dv = Dk); R is its S_T from S_0 = 0;
 * G is gdn_backward's dS_0 with dS_T = 0.  This call does the composition:
 *   out[b] = op(Phi[b]) S[b] + R[b]   for b < n,  op = identity or transpose
 *   Phi   device, fp32 [n, Dk, Dk] contiguous
 *   S     device, fp32 [n, Dk, Dv] contiguous
 *   R     device, fp32 [n, Dk, Dv] contiguous, or NULL (zero)
 *   out   device, fp32 [n, Dk, Dv] (written); may be R itself, must not overlap Phi or S
 *   transpose  0: Phi S + R;  1: Phi^T S + R
 * n at most 65535, Dk and Dv at most 4096; buffers 16-byte aligned.  Returns GDN_OK,
 * GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_MISALIGNED or GDN_ERR_CUDA. */
int gdn_state_compose(int32_t n, int32_t Dk, int32_t Dv, const float* Phi, const float* S,
                      const float* R, float* out, int32_t transpose, void* stream);

/* ---- KDA variant: a decay gate per key channel ------------------------------------------
 * The recurrence with the scalar gate g of a value head replaced by one gate per key
 * channel (the KDA module's decay, whose parameters a_log and b_alpha the dormouse "KDA
 * attention arm" page names):
 *   g[c] = exp(-exp(a_log[h]) * softplus(alpha[t, h*Dk + c] + b_alpha[h*Dk + c]))
 *   S_d = diag(g) S_{t-1};  kv = S_d^T k_hat;  delta = beta (v - kv)
 *   S_t = S_d + k_hat delta^T;  o_t = scale S_t^T q_hat
 * (q_hat, k_hat, beta and the key-head map as for gdn_forward).  Equal gates on every
 * channel give gdn_forward's recurrence.  This is its forward in token form, one token
 * after another per (sequence, value head): a decode step is a batch of one-token
 * sequences.
 * shape: as for gdn_forward (total_chunks and saved states are not used).
 *   q, k, v, o    device, as for gdn_forward (o written)
 *   alpha         device, fp32 [total_tokens, alpha_ld >= Hv*Dk]: channel c of value head
 *                 h at column h*Dk + c
 *   beta_raw      device, fp32 [total_tokens, beta_ld >= Hv]
 *   a_log         device, fp32 [Hv];  b_alpha  device, fp32 [Hv*Dk]
 *   cu_seqlens    device, int32 [n_seqs + 1] (token ranges are clamped to [0,
 *                 total_tokens))
 *   S_in          device, fp32 [n_seqs, Hv, Dk, Dv] or NULL (zero)
 *   S_out         device, fp32 [n_seqs, Hv, Dk, Dv] (written; may be S_in)
 * Needs no workspace.  Returns as gdn_decode_step does. */
int gdn_kda_forward(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                    int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                    int64_t alpha_ld, const float* beta_raw, int64_t beta_ld, const float* a_log,
                    const float* b_alpha, const int32_t* cu_seqlens, const float* S_in,
                    float* S_out, void* o, int64_t o_ld, void* stream);

/* gdn_kda_forward as a chunked prefill on the tensor cores (bf16 inputs, Dk and Dv in
 * {64, 128}): the same recurrence and outputs (o, S_out), formed chunk by chunk (C = 64
 * tokens) from the per-channel chunk algebra.  Per (chunk, value head), with l the
 * per-channel log gates and G their inclusive cumsum over the chunk's rows:
 *   A[r][s] = b_r sum_i k_r[i] k_s[i] e^{G_r[i] - G_s[i]} (s < r),  T = (I + A)^-1,
 *   P[r][s] = sum_i q_r[i] k_s[i] e^{G_r[i] - G_s[i]} (s <= r),
 *   W = T diag(b) (K e^G),  U = T diag(b) V,  Delta = U - W S,
 *   O = scale ((Q e^G) S + P Delta),  S' = diag(e^{G_last}) S + (K e^{G_last - G})^T Delta.
 * A and P are summed pair by pair over the channels on CUDA cores, so every exponent is
 * <= 0 however fast the gates decay; T, the products, the chunk walk and the output run
 * on the tensor cores (the walk carries S in fp32).
 * shape: as for gdn_forward (total_chunks and chunk_offsets from gdn_plan).
 * Arguments as gdn_kda_forward, plus chunk_offsets (device, int32 [n_seqs + 1]) and a
 * workspace of gdn_kda_forward_chunked_workspace_bytes(shape) bytes (256-byte aligned;
 * 0 for an unsupported shape).  Returns GDN_ERR_UNSUPPORTED for fp32 inputs or other head
 * sizes (use gdn_kda_forward), otherwise as gdn_forward. */
size_t gdn_kda_forward_chunked_workspace_bytes(const gdn_shape* shape);
int gdn_kda_forward_chunked(const gdn_shape* shape, const void* q, int64_t q_ld,
                            const void* k, int64_t k_ld, const void* v, int64_t v_ld,
                            const float* alpha, int64_t alpha_ld, const float* beta_raw,
                            int64_t beta_ld, const float* a_log, const float* b_alpha,
                            const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                            const float* S_in, float* S_out, void* o, int64_t o_ld,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Reverse mode of gdn_kda_forward, in token form: given dO and dS_T (NULL = zero) it
 * returns dq, dk (summed over the value heads that share a key head), dv, d alpha
 * [total_tokens, Hv*Dk], d beta_raw, d a_log [Hv], d b_alpha [Hv*Dk] (sums over every
 * token of every sequence) and dS_0 (NULL skips it).  All sums over value columns, value
 * heads and tokens are formed in a fixed order: results are bit-reproducible.
 * Each (sequence, value head, 32-column slice of the state) first walks its tokens
 * forward saving the state every 8 tokens, then walks them in reverse, recomputing each
 * 8-token segment from its saved state.  The workspace (16-byte aligned, at least
 * gdn_kda_backward_workspace_bytes(shape) bytes) holds those states and the per-slice
 * shares of dq_hat, dk_hat, dg, d beta: about (T/8 + n_seqs) * Hv * Dk * Dv * 4 +
 * T * Hv * (Dv/32) * (3 Dk + 1) * 4 bytes.
 * shape: as for gdn_kda_forward, with Dv >= 32.  Buffers and strides as there; dq, dk,
 * dv, dO have the dtype; dalpha and dbeta_raw are fp32 with strides >= Hv*Dk and >= Hv.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_MISALIGNED,
 * GDN_ERR_WORKSPACE or GDN_ERR_CUDA; nothing is launched on an error. */
size_t gdn_kda_backward_workspace_bytes(const gdn_shape* shape);
int gdn_kda_backward(const gdn_shape* shape, const void* q, int64_t q_ld, const void* k,
                     int64_t k_ld, const void* v, int64_t v_ld, const float* alpha,
                     int64_t alpha_ld, const float* beta_raw, int64_t beta_ld,
                     const float* a_log, const float* b_alpha, const int32_t* cu_seqlens,
                     const float* S0, const void* dO, int64_t dO_ld, const float* dS_T,
                     void* dq, int64_t dq_ld, void* dk, int64_t dk_ld, void* dv, int64_t dv_ld,
                     float* dalpha, int64_t dalpha_ld, float* dbeta_raw, int64_t dbeta_ld,
                     float* da_log, float* db_alpha, float* dS0, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Synchronises `stream` and returns the device-side status recorded in
 * `workspace` by the last gdn_forward / gdn_backward that used it (GDN_OK, or
 * the first device error), or GDN_ERR_CUDA if the stream itself failed. */
int gdn_read_device_status(const void* workspace, void* stream);

/* A static, human-readable name for a gdn_status value. */
const char* gdn_status_string(int status);

/* After a call of this host thread returned GDN_ERR_CUDA: which CUDA call
 * failed and the CUDA error name; "" otherwise.  The string is owned by the
 * library and stays valid until this thread's next gdn_forward / gdn_backward. */
const char* gdn_last_error(void);

/* Profiling aid (changes no result).  Between gdn_profile_begin and
 * gdn_profile_end, every kernel that gdn_forward / gdn_backward launch from the
 * calling host thread is bracketed by two of the caller's CUDA events, recorded
 * on the call's stream: launch i (counted from begin) records events[2*i] just
 * before and events[2*i+1] just after itself and stores its kernel id in
 * kernel_ids[i], for i < n_pairs.  `events` holds 2*n_pairs cudaEvent_t handles
 * created by the caller (plain events, not disabled timing); the caller reads
 * cudaEventElapsedTime(events[2i], events[2i+1]) after synchronising.  The
 * registration is per host thread and holds pointers only.
 * gdn_profile_begin returns GDN_OK or GDN_ERR_INVALID_ARG; gdn_profile_end
 * returns the number of launches seen (which may exceed n_pairs). */
int gdn_profile_begin(void* const* events, int32_t* kernel_ids, int32_t n_pairs);
int gdn_profile_end(void);

/* Name of a kernel id reported through gdn_profile_begin ("?" if unknown). */
const char* gdn_kernel_name(int32_t kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
