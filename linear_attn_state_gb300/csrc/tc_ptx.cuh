// Inline-PTX helpers for sm_103a: mbarriers, TMA tensor loads, tcgen05 MMA
// with tensor-memory accumulators, and the shared-memory operand layout the
// tensor cores read (K-major, 128-byte swizzle).
#pragma once

#include <cstdint>

#include <cuda.h>

namespace hypic {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

// One suspending poll: the thread may sleep (up to ~2 us) until the phase
// completes, without taking issue slots from the other warps.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 2000;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

// At most `limit` suspending polls of the barrier phase; false when it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try(bar, phase)) return true;
  return false;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Makes generic-proxy shared-memory writes visible to the async proxy
// (tensor cores, TMA).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05

// Warp-wide: allocates `ncols` tensor-memory columns, address written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16, single CTA.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define HYPIC_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define HYPIC_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                    "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 lanes x 32 consecutive columns: thread t of the warp receives lane
// (warp's lane quarter + t), columns [col, col + 32).
// 32 lanes x 16 consecutive columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : HYPIC_R8(0), HYPIC_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : HYPIC_R8(0), HYPIC_R8(8), HYPIC_R8(16), HYPIC_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      HYPIC_W8(0), HYPIC_W8(8), HYPIC_W8(16), HYPIC_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef HYPIC_R8
#undef HYPIC_W8

// ---------------------------------------------------------------- operand layout
//
// K-major, 128-byte swizzle, 16-bit elements: a tile is a stack of "K blocks"
// of 64 elements (128 bytes) along K; inside a K block row r (the M or N
// index) occupies 128 bytes at r*128, and its eight 16-byte chunks are
// permuted by XOR with (r mod 8).  Eight rows form a 1024-byte swizzle atom;
// tiles start 1024-byte aligned.  One MMA consumes K = 16 (32 bytes), so the
// descriptor of K step s inside a K block starts 32*s bytes into it.

// Byte offset of element (row, k) in a K-major SW128 tile with `rows` rows
// per K block.
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t k, uint32_t rows) {
  const uint32_t kb = k >> 6, kk = k & 63;
  return kb * rows * 128u + (row >> 3) * 1024u + (row & 7u) * 128u +
         ((((kk >> 3) ^ (row & 7u))) << 4) + ((kk & 7u) << 1);
}

// Byte offset of the 16-byte chunk holding elements (row, 8c .. 8c+7).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t row, uint32_t c8, uint32_t rows) {
  const uint32_t kb = c8 >> 3, cc = c8 & 7u;
  return kb * rows * 128u + (row >> 3) * 1024u + (row & 7u) * 128u + ((cc ^ (row & 7u)) << 4);
}

// Shared-memory matrix descriptor: K-major, SWIZZLE_128B, SBO = 1024 bytes
// (8-row group stride), tcgen05 descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                   // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                 // stride byte offset
  d |= 1ull << 46;                                              // version
  d |= 2ull << 61;                                              // SWIZZLE_128B
  return d;
}

// MN-major SW128 operand: element (mn, k) of a tile whose MN atoms (64 wide)
// are `lbo` bytes apart; K rows 128 bytes apart, 8-row groups 1024 apart.
__device__ __forceinline__ uint32_t mn_chunk(uint32_t mn8, uint32_t k, uint32_t lbo) {
  // 16-byte chunk holding elements (8*mn8 .. 8*mn8+7, k)
  return (mn8 >> 3) * lbo + (k >> 3) * 1024u + (k & 7u) * 128u + (((mn8 & 7u) ^ (k & 7u)) << 4);
}

__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo = 1024) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;   // MN-atom stride
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;   // 8-row K-group stride
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N) {
  return (1u << 4)                // D format: f32
         | (0u << 7)              // A format: f16
         | (0u << 10)             // B format: f16
         | (0u << 15)             // A K-major
         | (0u << 16)             // B K-major
         | ((N >> 3) << 17)       // N / 8
         | ((M >> 4) << 24);      // M / 16
}

}  // namespace tc
}  // namespace hypic
