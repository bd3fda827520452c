// gdn_tc.cuh -- CTA-level helpers for the tensor-core (tcgen05) kernels:
// accumulator row ownership, epilogue column walks, staging of bf16 operand
// tiles in the K-major 128B-swizzled layout, and MMA completion waits that all
// threads agree on.
#pragma once

#include "gdn_device.cuh"
#include "umma.cuh"

namespace gdn {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Threads per CTA of the tensor-core kernels: 16 warps, so that each TMEM lane
// quarter (warps w, w + 4, w + 8, w + 12) is read by kGroups warps that split an
// accumulator's columns between them.
constexpr int kTcThreads = 512;
constexpr int kGroups = kTcThreads / 128;
__device__ __forceinline__ int col_group() { return (int)(threadIdx.x >> 7); }

// The first kCtlBytes of a tensor-core kernel's (1024-aligned) shared memory: its
// mbarriers and the TMEM address, at the same place whatever role the CTA plays.
constexpr uint32_t kCtlBytes = 1024;
struct CtaCtl {
  uint64_t bar[8];
  uint32_t tmem;
};
// All threads: nbar mbarriers (arrival count 1) and ncols TMEM columns.
__device__ __forceinline__ void cta_setup(CtaCtl* ctl, int nbar, uint32_t ncols) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nbar; ++i) tc::mbar_init(&ctl->bar[i], 1);
    tc::fence_mbar_init();
  }
  if ((threadIdx.x >> 5) == 0) {
    tc::tmem_alloc(&ctl->tmem, ncols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}
__device__ __forceinline__ void cta_teardown(CtaCtl* ctl, uint32_t ncols) {
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if ((threadIdx.x >> 5) == 0) tc::tmem_dealloc(ctl->tmem, ncols);
}

// A batch's cu_seqlens and chunk offsets copied into shared memory for a CTA's chunk
// lookups (each a global round trip otherwise, on the path of the thread that issues
// the copies), when the batch has fewer than `cap` sequences.
struct SeqTab {
  const int32_t* cu;
  const int32_t* coff;
};
// All threads, then a CTA barrier: fills the cache at `sm` (2 cap int32) if the batch
// fits, and returns the table to read.
__device__ __forceinline__ SeqTab seq_tab(const Params& p, int32_t* sm, int cap) {
  const int m = p.n_seqs + 1;
  const bool fits = m <= cap;
  if (fits)
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      sm[i] = p.cu[i];
      sm[cap + i] = p.coff[i];
    }
  __syncthreads();
  return fits ? SeqTab{sm, sm + cap} : SeqTab{p.cu, p.coff};
}
__device__ __forceinline__ bool chunk_info(const Params& p, const SeqTab& tab, int c, int* n,
                                           int64_t* t0, int* len) {
  return chunk_info_at(tab.cu, tab.coff, p.n_seqs, p.NC, p.T, c, n, t0, len);
}

// Readiness flags between the CTAs of one cooperative launch (all co-resident).
// The producer publishes after every write of the unit has completed (its bulk
// stores waited for, a CTA barrier, then this call on one thread); the consumer
// acquires before issuing bulk copies that read the unit's outputs.
__device__ __forceinline__ void publish_flag(uint32_t* flag) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(1u) : "memory");
}
// publish_flag for several units whose writes are all done: one fence for all of them,
// then a relaxed store per flag (the fence and a later store form the release), at
// flags + i * stride for i < count.
__device__ __forceinline__ void publish_flags(uint32_t* flags, size_t stride, int count) {
  if (count <= 0) return;
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  for (int i = 0; i < count; ++i)
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flags + (size_t)i * stride), "r"(1u)
                 : "memory");
}
// A relaxed read of a counter or flag (no ordering: for heuristics only).
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* flag) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* flag) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v;
}
// How long a wait on another CTA's readiness flag may take before it gives up and
// records GDN_ERR_TIMEOUT (wall time, ns).  A build with 0 makes every wait that is not
// satisfied at once run out, which is how the failure path is tested.
#ifndef GDN_FLAG_WAIT_LIMIT_NS
#define GDN_FLAG_WAIT_LIMIT_NS 2000000000ull
#endif
// One thread: true once *flag is set; false if it is still clear after
// GDN_FLAG_WAIT_LIMIT_NS (2 s).
__device__ __forceinline__ bool flag_ready(const uint32_t* flag) {
  return ld_acquire(flag) != 0u;
}
__device__ __forceinline__ bool wait_flag(const uint32_t* flag) {
  bool ok = flag_ready(flag);
  if (!ok) {
    const uint64_t t0 = tc::globaltimer_ns();
    while (!(ok = flag_ready(flag))) {
      __nanosleep(128);
      if (tc::globaltimer_ns() - t0 > (uint64_t)(GDN_FLAG_WAIT_LIMIT_NS)) break;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return ok;
}

// Accumulator row held by this thread's TMEM lane for an M-row MMA, or -1.
// M = 128: warp w (mod 4) owns rows 32w..32w+31 (row = lane).  M = 64: rows
// 16w..16w+15 sit in lanes 32w..32w+15 (checked by tests/test_umma_layout.py).
__device__ __forceinline__ int acc_row(int M) {
  const int w = (threadIdx.x >> 5) & 3, l = threadIdx.x & 31;
  if (M == 128) return 32 * w + l;
  return l < 16 ? 16 * w + l : -1;
}
__device__ __forceinline__ uint32_t lane_quarter() {
  return (uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16;
}

// Walks the accumulator columns [0, N) in 16-column pieces; the kGroups warps that
// share a lane quarter take every kGroups-th piece.  f(row, col0, v[16]) runs for
// rows < valid.  Whole warps must call this.
template <class F>
__device__ __forceinline__ void acc_walk(uint32_t tmem, int M, int N, int valid, F f) {
  const int row = acc_row(M);
  for (int c = col_group() * 16; c < N; c += 16 * kGroups) {
    float v[16];
    tc::tmem_ld16(tmem + lane_quarter() + (uint32_t)c, v);
    tc::tmem_ld_wait();
    if (row >= 0 && row < valid) f(row, c, v);
  }
}

// M = 64 accumulators read with the 16x32bx2 loads, which hand both halves of a warp
// the quarter's 16 live lanes: thread t of warp w holds row 16 (w % 4) + (t % 16), and
// threads 16-31 take the second column piece of each load.
__device__ __forceinline__ int x2_row() {
  return 16 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 15);
}
__device__ __forceinline__ int x2_half() { return (threadIdx.x >> 4) & 1; }

// Walks the columns [0, N) of an M = 64 accumulator in 16-column pieces, two per load:
// the kGroups warps of a lane quarter take pieces grp + 2 kGroups i (threads 0-15) and
// grp + kGroups (2i + 1) (threads 16-31).  f(row, col0, v[16]) runs for rows < valid.
// The loads may read up to 16 kGroups + 15 columns past N (allocated TMEM, ignored).
// Whole warps must call this.
template <class F>
__device__ __forceinline__ void acc_walk64(uint32_t tmem, int N, int valid, F f) {
  const int row = x2_row(), half = x2_half();
  for (int c = col_group() * 16; c < N; c += 32 * kGroups) {
    float v[16];
    tc::tmem_ld16_x2<16 * kGroups>(tmem + lane_quarter() + (uint32_t)c, v);
    tc::tmem_ld_wait();
    const int col = c + half * 16 * kGroups;
    if (row < valid && col < N) f(row, col, v);
  }
}
// As acc_walk64 in 8-column halves of each warp's 16-column piece (for N <= 16 kGroups):
// threads 0-15 take columns [c, c + 8), threads 16-31 [c + 8, c + 16); f(row, col0, v[8]).
template <class F>
__device__ __forceinline__ void acc_walk64_8(uint32_t tmem, int N, int valid, F f) {
  const int row = x2_row(), half = x2_half();
  for (int c = col_group() * 16; c < N; c += 16 * kGroups) {
    float v[8];
    tc::tmem_ld8_x2<8>(tmem + lane_quarter() + (uint32_t)c, v);
    tc::tmem_ld_wait();
    const int col = c + half * 8;
    if (row < valid && col < N) f(row, col, v);
  }
}
// Sum of a per-thread value over the two threads that hold the same x2 row.
__device__ __forceinline__ float x2_pair_sum(float v) {
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// Stages a bf16 K-major SW128 tile of rows x cols (cols a multiple of 8) from
// f(r, c) -> float, 8 elements (one 16-byte store) per step.
template <class F>
__device__ __forceinline__ void stage_tile(uint8_t* tile, int rows, int cols, F f) {
  const int cpr = cols >> 3;
  for (int idx = threadIdx.x; idx < rows * cpr; idx += blockDim.x) {
    const int r = idx / cpr, c8 = (idx - (idx / cpr) * cpr) << 3;
    __align__(16) __nv_bfloat162 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __floats2bfloat162_rn(f(r, c8 + 2 * u), f(r, c8 + 2 * u + 1));
    *(uint4*)(tile + tc::sw128_offset(r, c8, rows)) = *(const uint4*)v;
  }
}

// Stages an fp32 row-major source M (R rows x Cc columns, row stride ld floats,
// 16-byte aligned rows, Cc a multiple of 8) into a natural tile tn (R rows, Cc
// columns) and / or a transposed tile tt (Cc rows, R columns; tt_rows = its row
// count); element (r, c) is multiplied by rs(r) * cs(c).  Rows r >= valid read as
// zero.  Consecutive threads take consecutive source rows, so that the
// transposed writes of a warp land in one tile row (no bank conflicts) and the
// natural 16-byte writes of 8 threads cover all 32 banks.
template <class RS, class CS>
__device__ __forceinline__ void stage_f32(const float* M, int R, int Cc, int64_t ld, int valid,
                                          uint8_t* tn, uint8_t* tt, int tt_rows, RS rs, CS cs) {
  const int cpr = Cc >> 3, total = R * cpr;
  // four items per thread per batch: all loads are issued before any store
  for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
    float4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * blockDim.x;
      const int r = idx % R, c0 = (idx / R) << 3;
      a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < total && r < valid) {
        a[u] = *(const float4*)(M + (int64_t)r * ld + c0);
        b[u] = *(const float4*)(M + (int64_t)r * ld + c0 + 4);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx >= total) break;
      const int r = idx % R, c0 = (idx / R) << 3;
      const float s = r < valid ? rs(r) : 0.f;
      float v[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= s * cs(c0 + e);
      if (tn) {
        __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        *(uint4*)(tn + tc::sw128_offset(r, c0, R)) = *(const uint4*)pk;
      }
      if (tt)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *(__nv_bfloat16*)(tt + tc::sw128_offset(c0 + e, r, tt_rows)) = __float2bfloat16_rn(v[e]);
    }
  }
}
struct One {
  __device__ __forceinline__ float operator()(int) const { return 1.f; }
};

// As stage_f32 for a bf16 row-major source (row stride ld elements, 16-byte
// aligned rows).  Outputs: tn (natural, unscaled, tn_rows rows), tn2 (natural,
// scaled by rs(r), R rows), tt (transposed, scaled by rs(r), tt_rows rows).
template <class RS>
__device__ __forceinline__ void stage_bf16(const __nv_bfloat16* M, int R, int Cc, int64_t ld,
                                           int valid, uint8_t* tn, int tn_rows, uint8_t* tn2,
                                           uint8_t* tt, int tt_rows, RS rs) {
  const int cpr = Cc >> 3, total = R * cpr;
  for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * blockDim.x;
      const int r = idx % R, c0 = (idx / R) << 3;
      raw[u] = make_uint4(0, 0, 0, 0);
      if (idx < total && r < valid) raw[u] = *(const uint4*)(M + (int64_t)r * ld + c0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx >= total) break;
      const int r = idx % R, c0 = (idx / R) << 3;
      if (tn) *(uint4*)(tn + tc::sw128_offset(r, c0, tn_rows)) = raw[u];
      if (tn2 || tt) {
        const __nv_bfloat16* e = (const __nv_bfloat16*)&raw[u];
        const float s = rs(r);
        if (tn2) {
          __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            pk[q] = __floats2bfloat162_rn(__bfloat162float(e[2 * q]) * s,
                                          __bfloat162float(e[2 * q + 1]) * s);
          *(uint4*)(tn2 + tc::sw128_offset(r, c0, R)) = *(const uint4*)pk;
        }
        if (tt)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *(__nv_bfloat16*)(tt + tc::sw128_offset(c0 + q, r, tt_rows)) =
                __float2bfloat16_rn(__bfloat162float(e[q]) * s);
      }
    }
  }
}

// Writes 16 consecutive elements v[0..15] of row r, columns c0..c0+15 (c0 a
// multiple of 16), of a K-major SW128 bf16 tile with two 16-byte stores.
__device__ __forceinline__ void tile_put16(uint8_t* tile, int rows, int r, int c0, const float* v) {
  __align__(16) __nv_bfloat162 pk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pk[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
  *(uint4*)(tile + tc::sw128_offset(r, c0, rows)) = ((const uint4*)pk)[0];
  *(uint4*)(tile + tc::sw128_offset(r, c0 + 8, rows)) = ((const uint4*)pk)[1];
}

// Reads 16 consecutive elements of row r, columns c0..c0+15, of a SW128 bf16 tile.
__device__ __forceinline__ void tile_get16(const uint8_t* tile, int rows, int r, int c0, float* v) {
  const uint4 a = *(const uint4*)(tile + tc::sw128_offset(r, c0, rows));
  const uint4 b = *(const uint4*)(tile + tc::sw128_offset(r, c0 + 8, rows));
  const __nv_bfloat16* ea = (const __nv_bfloat16*)&a;
  const __nv_bfloat16* eb = (const __nv_bfloat16*)&b;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = __bfloat162float(ea[j]);
    v[8 + j] = __bfloat162float(eb[j]);
  }
}

// 8 consecutive elements (c0 a multiple of 8): one 16-byte chunk of a SW128 bf16 tile.
__device__ __forceinline__ void tile_put8(uint8_t* tile, int rows, int r, int c0, const float* v) {
  __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) pk[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
  *(uint4*)(tile + tc::sw128_offset(r, c0, rows)) = *(const uint4*)pk;
}
__device__ __forceinline__ void tile_get8(const uint8_t* tile, int rows, int r, int c0, float* v) {
  const uint4 a = *(const uint4*)(tile + tc::sw128_offset(r, c0, rows));
  const __nv_bfloat16* ea = (const __nv_bfloat16*)&a;
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __bfloat162float(ea[j]);
}

// Reads one bf16 element of a K-major SW128 tile as float.
__device__ __forceinline__ float tile_get(const uint8_t* tile, int rows, int r, int c) {
  return __bfloat162float(*(const __nv_bfloat16*)(tile + tc::sw128_offset(r, c, rows)));
}

// Stores one bf16 element of a K-major SW128 tile.
__device__ __forceinline__ void tile_put(uint8_t* tile, int rows, int r, int c, float x) {
  *(__nv_bfloat16*)(tile + tc::sw128_offset(r, c, rows)) = __float2bfloat16_rn(x);
}

// Copies `bytes` (multiple of 16) between 16-byte-aligned buffers with the whole CTA.
__device__ __forceinline__ void cta_copy16(void* dst, const void* src, uint32_t bytes) {
  uint4* d = (uint4*)dst;
  const uint4* s = (const uint4*)src;
  for (uint32_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) d[i] = s[i];
}

// Thread 0 issues MMAs through `issue()`, commits them onto `bar`, and every
// thread waits.  Returns false on every thread if any thread's bounded wait ran
// out (the status word then holds GDN_ERR_TIMEOUT).  Writers of the operand
// tiles must have called tc::fence_async_smem() before this.
template <class F>
__device__ __forceinline__ bool mma_run(F issue, uint64_t* bar, uint32_t& phase,
                                        DeviceStatus* status, int detail) {
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc::fence_after_sync();
    issue();
    tc::mma_commit(bar);
  }
  const bool ok = tc::mbar_wait(bar, phase);
  phase ^= 1u;
  tc::fence_after_sync();
  const int bad = __syncthreads_or(ok ? 0 : 1);
  if (bad && threadIdx.x == 0) set_status(status, GDN_ERR_TIMEOUT, detail);
  return bad == 0;
}

// mma_run in two halves, for work that overlaps the tensor core: mma_issue
// (all threads: barrier, then thread 0 issues and commits onto `bar`) and
// mma_wait (all threads: bounded wait, then a barrier that agrees on the outcome).
template <class F>
__device__ __forceinline__ void mma_issue(F issue, uint64_t* bar) {
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc::fence_after_sync();
    issue();
    tc::mma_commit(bar);
  }
}
__device__ __forceinline__ bool mma_wait(uint64_t* bar, uint32_t& phase, DeviceStatus* status,
                                         int detail) {
  const bool ok = tc::mbar_wait(bar, phase);
  phase ^= 1u;
  tc::fence_after_sync();
  const int bad = __syncthreads_or(ok ? 0 : 1);
  if (bad && threadIdx.x == 0) set_status(status, GDN_ERR_TIMEOUT, detail);
  return bad == 0;
}

}  // namespace gdn
