// umma.cuh -- Blackwell (sm_100 family) tensor-core building blocks in inline PTX:
// TMEM allocation, tcgen05.mma (kind::f16, bf16 x bf16 -> fp32), tcgen05.commit
// onto an mbarrier, tcgen05.ld of the fp32 accumulator, shared-memory matrix
// descriptors for K-major operands in the 128-byte swizzled layout, and bounded
// mbarrier waits.
//
// Operand tiles ("K-major SW128"): a tile of R rows (the M or N index) by K
// columns of bf16 is stored as K/64 column blocks; block b holds columns
// [64b, 64b+64) of every row, row r at byte r*128 of the block, and the 16-byte
// chunk j of a row at chunk position j ^ (r % 8).  Blocks are R*128 bytes
// apart and 1024-byte aligned.  This is the layout the MMA unit reads with a
// descriptor of swizzle mode 128B, stride between 8-row groups 1024 bytes; a
// K step of 16 elements inside a block advances the descriptor's start
// address by 32 bytes.
//
// Accumulator (M = 128, cta_group::1): row i of D lives in TMEM lane i, column
// j in TMEM column (base + j), one fp32 per cell.  Warp w of a CTA may read
// lanes [32 (w % 4), 32 (w % 4) + 32).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up after
// `limit_ns` nanoseconds of wall time and returns false (the caller records
// GDN_ERR_TIMEOUT and winds down); never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < (1u << 30); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Raises the transaction count of the current phase without arriving (a later
// arrive_expect_tx by the same thread completes the arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads operands through it).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- TMEM
// Whole warp: allocates `ncols` TMEM columns (power of two, >= 32) and writes
// the base address to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Whole warp: 16 consecutive fp32 columns of the warp's 32 lanes; thread t gets
// lane (lane base + t).  Follow with tmem_ld_wait() before using the values.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Whole warp, for M = 64 accumulators (rows in lanes 0-15 of each quarter): lane t
// of the warp's first 16 lanes goes to thread t with columns [taddr, taddr + 16) and
// to thread t + 16 with columns [taddr + OFF, taddr + OFF + 16), so every thread holds
// 16 consecutive values of one row.  Follow with tmem_ld_wait().
template <int OFF>
__device__ __forceinline__ void tmem_ld16_x2(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(OFF));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// As tmem_ld16_x2 with 8 columns per thread.
template <int OFF>
__device__ __forceinline__ void tmem_ld8_x2(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr), "n"(OFF));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ descriptors
// Shared-memory descriptor of a K-major, 128-byte-swizzled operand starting at
// shared address `saddr` (the block base must be 1024-byte aligned; the start
// may be offset by a multiple of 32 bytes inside the first 128-byte row for
// K steps).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading-dimension byte offset (unused with SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8-row groups are 1024 B apart
  d |= (uint64_t)1 << 46;              // descriptor version for sm_100 family
  d |= (uint64_t)2 << 61;              // swizzle mode: 128B
  return d;
}

// Shared-memory descriptor of an MN-major, 128-byte-swizzled operand: the tile
// is stored with one 128-byte row per K index holding 64 consecutive M (or N)
// elements, 8 rows to a 1024-byte swizzle atom.  `mn_stride` is the byte
// distance between consecutive 64-element MN blocks (leading-dimension byte
// offset); consecutive 8-row K groups are 1024 B apart (stride byte offset).
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator,
// shape M x N; a_mn / b_mn select MN-major (transposed) storage of A / B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false,
                                                  bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One thread: D[tmem] (+)= A * B^T, single K=16 step.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One thread: arrive once on `bar` when every MMA this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Byte offset of element (row, k) in a K-major SW128 bf16 tile of `rows` rows.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
  const uint32_t blk = (uint32_t)(k >> 6);
  const uint32_t byte = (uint32_t)(k & 63) * 2u;
  const uint32_t chunk = (byte >> 4) ^ (uint32_t)(row & 7);
  return blk * (uint32_t)rows * 128u + (uint32_t)row * 128u + chunk * 16u + (byte & 15u);
}

// Issues D (+)= A[M x K] * B[N x K]^T over K (multiple of 16) from K-major SW128
// tiles at shared addresses a_base (M rows) and b_base (N rows).  a_pitch /
// b_pitch are the byte distances between consecutive 64-column blocks of each
// tile (rows * 128 for a tile stored on its own).
__device__ __forceinline__ void mma_tile_p(uint32_t d_tmem, uint32_t a_base, uint32_t a_pitch,
                                           int M, uint32_t b_base, uint32_t b_pitch, int N,
                                           int K, uint32_t accumulate_first) {
  const uint32_t idesc = idesc_bf16(M, N);
  for (int kk = 0; kk < K; kk += 16) {
    const uint32_t a = a_base + (uint32_t)(kk >> 6) * a_pitch + (uint32_t)(kk & 63) * 2u;
    const uint32_t b = b_base + (uint32_t)(kk >> 6) * b_pitch + (uint32_t)(kk & 63) * 2u;
    mma_bf16(d_tmem, desc_sw128(a), desc_sw128(b), idesc, (kk > 0) ? 1u : accumulate_first);
  }
}
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_base, int M, uint32_t b_base,
                                         int N, int K, uint32_t accumulate_first) {
  mma_tile_p(d_tmem, a_base, (uint32_t)M * 128u, M, b_base, (uint32_t)N * 128u, N, K,
             accumulate_first);
}

// As mma_tile_p with either operand optionally MN-major.  An MN-major operand
// X (M or N = 64 or 128) is a SW128 tile stored as rows = K indices (its
// K-major view transposed): element (mn, k) at sw128_offset(k, mn, x_rows),
// with x_rows >= K the tile's row count; its 64-element MN blocks are
// x_rows * 128 bytes apart, and a K step of 16 advances 16 rows (2048 bytes).
// A K-major operand keeps the meaning of mma_tile_p (pitch between 64-column
// blocks).
__device__ __forceinline__ void mma_tile_x(uint32_t d_tmem, uint32_t a_base, bool a_mn,
                                           uint32_t a_pitch, int M, uint32_t b_base, bool b_mn,
                                           uint32_t b_pitch, int N, int K,
                                           uint32_t accumulate_first) {
  const uint32_t idesc = idesc_bf16(M, N, a_mn, b_mn);
  for (int kk = 0; kk < K; kk += 16) {
    const uint64_t da =
        a_mn ? desc_sw128_mn(a_base + (uint32_t)kk * 128u, a_pitch)
             : desc_sw128(a_base + (uint32_t)(kk >> 6) * a_pitch + (uint32_t)(kk & 63) * 2u);
    const uint64_t db =
        b_mn ? desc_sw128_mn(b_base + (uint32_t)kk * 128u, b_pitch)
             : desc_sw128(b_base + (uint32_t)(kk >> 6) * b_pitch + (uint32_t)(kk & 63) * 2u);
    mma_bf16(d_tmem, da, db, idesc, (kk > 0) ? 1u : accumulate_first);
  }
}

// Bytes of a K-major SW128 bf16 tile of `rows` rows and `cols` columns.
__host__ __device__ __forceinline__ uint32_t sw128_bytes(int rows, int cols) {
  return (uint32_t)((cols + 63) / 64) * (uint32_t)rows * 128u;
}

// ------------------------------------------------------------ TMA tiles
// One thread: loads the box at (x, y) (x = column, a multiple of 8 bf16; y =
// row) of the 2-D tensor map into shared memory; completion is signalled on
// `bar` through its transaction count.  The map lives in kernel-parameter
// space (__grid_constant__).
// Brings a tensor map (the generic address of a __grid_constant__ kernel parameter) into
// the descriptor cache ahead of the copies that use it.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tmap) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------ bulk copies
// One thread: copies `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global memory into shared memory with the bulk-copy engine; completion
// is signalled on `bar` through its transaction count.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One thread: copies `bytes` (multiple of 16; both addresses 16-byte aligned)
// from shared to global memory with the bulk-copy engine, in this thread's
// current bulk group.  Writers of the source must have run fence_async_smem()
// and synchronised with the issuing thread first.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
// One thread: asks for `bytes` (multiple of 16; 16-byte aligned address) of global
// memory to be brought into the L2 cache ahead of their use; no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gmem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem_src), "r"(bytes)
               : "memory");
}
// Closes the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk groups still read their shared
// memory source (the source may then be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of this thread's bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------- per-thread async copies
// One thread: copies 4 (16) bytes from global to shared memory without holding a
// register; the data is visible to this thread after cp_async_wait_all() and to
// the CTA after a barrier that follows it.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
// Closes this thread's current group of cp.async copies.
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's cp.async groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

}  // namespace tc
}  // namespace gdn
