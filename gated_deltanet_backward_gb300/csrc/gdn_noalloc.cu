// gdn_noalloc.cu -- gdn_forward for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: code that runs under a
// device-memory budget fixed when the process starts, plugin hosts that hand a
// kernel its inputs and outputs but no scratch buffer, and latency-sensitive
// paths that cannot accept the implicit device synchronisation of
// cudaMalloc / cudaFree.  For them the forward's scratch lives in one
// statically sized device array that the library carries with it.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)GDN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  Every GPU that loads this library holds it until the
// process exits.  In host code `g_scratch` only stands in for the symbol; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  Outside stream capture it is
// looked up again on every call (cudaGetSymbolAddress, with that device current): a
// device reset reloads the module and another context of the same device maps the
// array elsewhere, so an address kept from an earlier call can be stale.  While
// `stream` is capturing, the address of this device's last call outside capture is
// used (a symbol lookup can load the module, which capture does not allow); a first
// call on a device inside capture is refused.
int scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (!g_scratch_ptr[dev]) {
    return GDN_ERR_UNSUPPORTED;
  }
  *out = g_scratch_ptr[dev];
  return GDN_OK;
}

}  // namespace

namespace gdn {
void set_last_error(const char* msg);
}

extern "C" int gdn_forward_noalloc(const gdn_shape* s, const void* q, int64_t q_ld,
                                   const void* k, int64_t k_ld, const void* v, int64_t v_ld,
                                   const float* alpha, int64_t alpha_ld, const float* beta_raw,
                                   int64_t beta_ld, const float* a_log, const float* dt_bias,
                                   const int32_t* cu_seqlens, const int32_t* chunk_offsets,
                                   const float* S0, void* o, int64_t o_ld, float* S_T,
                                   void* saved_states, void* stream) {
  const size_t need = gdn_workspace_bytes(s, 0);
  if (need == 0)  // invalid shape: let the regular entry point name the problem
    return gdn_forward(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                       dt_bias, cu_seqlens, chunk_offsets, S0, o, o_ld, S_T, saved_states,
                       nullptr, 0, 0u, stream);
  if (need > kScratchBytes) {
    gdn::set_last_error(
        "gdn_forward_noalloc: this shape needs more scratch than the built-in "
        "GDN_NOALLOC_SCRATCH_BYTES; use gdn_forward with a caller workspace");
    return GDN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int rc = scratch_address((cudaStream_t)stream, &scratch);
  if (rc != GDN_OK) {
    gdn::set_last_error(rc == GDN_ERR_UNSUPPORTED
                            ? "gdn_forward_noalloc: first call on this device inside a stream "
                              "capture (call it once outside capture first)"
                            : "gdn_forward_noalloc: cudaGetSymbolAddress of the scratch failed");
    return rc;
  }
  // The scratch's status word is cleared by gdn_forward itself; every other
  // region is fully written before it is read.
  return gdn_forward(s, q, q_ld, k, k_ld, v, v_ld, alpha, alpha_ld, beta_raw, beta_ld, a_log,
                     dt_bias, cu_seqlens, chunk_offsets, S0, o, o_ld, S_T, saved_states,
                     scratch, kScratchBytes, 0u, stream);
}
