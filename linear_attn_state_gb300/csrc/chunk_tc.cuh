// Device helpers shared by the chunked tcgen05 segment builds (gated delta and
// KDA): operand packing and bf16 hi/lo splits, groups of MMAs issued from one
// asm block, named barriers, and the small fp32 shared-memory products of the
// 64x64 unit-triangular inverse.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"

namespace hypic {
namespace chunk {

using namespace tc;

// (a, b) -> fp16x2 with round-to-nearest-even, one packed conversion
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// bf16 hi/lo split of a pair by truncation: hi = the upper 16 bits of x
// (exact), lo = the upper 16 bits of x - hi (x - hi is exact in fp32), so
// hi + lo keeps 16 significant bits.  Element a in the low half of each word.
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  hi = __byte_perm(ua, ub, 0x7632);
  const float ra = a - __uint_as_float(ua & 0xFFFF0000u);
  const float rb = b - __uint_as_float(ub & 0xFFFF0000u);
  lo = __byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x7632);
}

// instruction descriptor bits on top of idesc_f16: operand majors and bf16 inputs
constexpr uint32_t ID_KK = 0;                 // A K-major, B K-major
constexpr uint32_t ID_KM = 1u << 16;          // A K-major (or tensor memory), B MN-major
constexpr uint32_t ID_MM = (1u << 15) | (1u << 16);
constexpr uint32_t ID_BF16 = (1u << 7) | (1u << 10);   // A and B bf16

// Eight MMAs into one accumulator from one asm block: operand i is the base
// descriptor (or tensor-memory address) plus the compile-time increment Ai / Bi
// (descriptor increments are byte offsets / 16), so each MMA costs two adds
// besides itself.  The first accumulates when acc0 != 0, the others always.
template <int A0, int A1, int A2, int A3, int A4, int A5, int A6, int A7, int B0, int B1, int B2,
          int B3, int B4, int B5, int B6, int B7>
__device__ __forceinline__ void mma8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 x, y;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, %4, %4;\n"
      " add.s64 x, %1, %5;\n add.s64 y, %2, %13;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, p;\n"
      " add.s64 x, %1, %6;\n add.s64 y, %2, %14;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %7;\n add.s64 y, %2, %15;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %8;\n add.s64 y, %2, %16;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %9;\n add.s64 y, %2, %17;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %10;\n add.s64 y, %2, %18;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %11;\n add.s64 y, %2, %19;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %12;\n add.s64 y, %2, %20;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      "}"
      :
      : "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc0), "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(A4),
        "n"(A5), "n"(A6), "n"(A7), "n"(B0), "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6),
        "n"(B7)
      : "memory");
}
// the same with A in tensor memory (all eight accumulate)
template <int A0, int A1, int A2, int A3, int A4, int A5, int A6, int A7, int B0, int B1, int B2,
          int B3, int B4, int B5, int B6, int B7>
__device__ __forceinline__ void mma8_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id) {
  const uint32_t acc0 = 1;
  asm volatile(
      "{\n .reg .pred q;\n .reg .b32 t;\n .reg .b64 y;\n setp.eq.b32 q, %4, %4;\n"
      " add.u32 t, %1, %5;\n add.s64 y, %2, %13;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %6;\n add.s64 y, %2, %14;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %7;\n add.s64 y, %2, %15;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %8;\n add.s64 y, %2, %16;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %9;\n add.s64 y, %2, %17;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %10;\n add.s64 y, %2, %18;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %11;\n add.s64 y, %2, %19;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %12;\n add.s64 y, %2, %20;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      "}"
      :
      : "r"(d), "r"(a), "l"(b), "r"(id), "r"(acc0), "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(A4),
        "n"(A5), "n"(A6), "n"(A7), "n"(B0), "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6),
        "n"(B7)
      : "memory");
}

// Four MMAs into one accumulator (all four accumulate), operands as in mma8_ss:
// the third product of a hi/lo pair of splits (the lo x lo product is dropped).
template <int A0, int A1, int A2, int A3, int B0, int B1, int B2, int B3>
__device__ __forceinline__ void mma4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id) {
  const uint32_t acc0 = 1;
  asm volatile(
      "{\n .reg .pred q;\n .reg .b64 x, y;\n setp.eq.b32 q, %4, %4;\n"
      " add.s64 x, %1, %5;\n add.s64 y, %2, %9;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %6;\n add.s64 y, %2, %10;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %7;\n add.s64 y, %2, %11;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      " add.s64 x, %1, %8;\n add.s64 y, %2, %12;\n tcgen05.mma.cta_group::1.kind::f16 [%0], x, y, %3, q;\n"
      "}"
      :
      : "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc0), "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(B0),
        "n"(B1), "n"(B2), "n"(B3)
      : "memory");
}
// the same with A in tensor memory
template <int A0, int A1, int A2, int A3, int B0, int B1, int B2, int B3>
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id) {
  const uint32_t acc0 = 1;
  asm volatile(
      "{\n .reg .pred q;\n .reg .b32 t;\n .reg .b64 y;\n setp.eq.b32 q, %4, %4;\n"
      " add.u32 t, %1, %5;\n add.s64 y, %2, %9;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %6;\n add.s64 y, %2, %10;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %7;\n add.s64 y, %2, %11;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      " add.u32 t, %1, %8;\n add.s64 y, %2, %12;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [t], y, %3, q;\n"
      "}"
      :
      : "r"(d), "r"(a), "l"(b), "r"(id), "r"(acc0), "n"(A0), "n"(A1), "n"(A2), "n"(A3), "n"(B0),
        "n"(B1), "n"(B2), "n"(B3)
      : "memory");
}

// 32 lanes x 16 consecutive columns store
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}


__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Role-wide OR of a predicate (named barrier with reduction).
__device__ __forceinline__ bool named_or(uint32_t id, uint32_t n, bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, o;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred o, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, o;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// C = alpha * A * B for small fp32 matrices in shared memory (row strides in
// floats).  `nt` consecutive threads starting at t = 0 share the work; thread t
// computes an RT x 4 output tile, so each k step is one 16-byte load of B and
// RT loads of A feeding 4 * RT independent FMAs.
template <int M, int N, int K, int RT>
__device__ __forceinline__ void smem_gemm(float* C, int ldc, const float* A, int lda,
                                          const float* B, int ldb, float alpha, int t) {
  constexpr int TN = N / 4;
  const int r0 = (t / TN) * RT, c0 = (t % TN) * 4;
  float acc[RT][4];
#pragma unroll
  for (int i = 0; i < RT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int m = 0; m < K; ++m) {
    const float4 b = *reinterpret_cast<const float4*>(B + m * ldb + c0);
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const float a = A[(r0 + i) * lda + m];
      acc[i][0] = fmaf(a, b.x, acc[i][0]);
      acc[i][1] = fmaf(a, b.y, acc[i][1]);
      acc[i][2] = fmaf(a, b.z, acc[i][2]);
      acc[i][3] = fmaf(a, b.w, acc[i][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < RT; ++i)
    *reinterpret_cast<float4*>(C + (r0 + i) * ldc + c0) =
        make_float4(alpha * acc[i][0], alpha * acc[i][1], alpha * acc[i][2], alpha * acc[i][3]);
}

// C = alpha * A * B for 32x32 fp32 matrices in shared memory, on 256 threads:
// four k-groups of 64 threads (k in [8 kg, 8 kg + 8)), each thread a 4x4 tile
// (float4 loads of 4 A rows and 4 B rows per 4 k, 64 independent FMAs),
// partial sums through the scratch P [4][32][32], then every thread sums one
// float4 of the result.  A k-group whose k-range lies where the lower-
// triangular operand is zero (B: k < column, A: k > row) skips its tile.
template <bool B_LOWER, bool A_LOWER>
__device__ __forceinline__ void gemm32_ksplit(float* C, int ldc, const float* A, int lda,
                                              const float* B, int ldb, float alpha, float* P,
                                              int t, uint32_t nb) {
  const int kg = t >> 6, tile = t & 63;
  const int r0 = (tile >> 3) * 4, c0 = (tile & 7) * 4, k0 = 8 * kg;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const bool skip = (B_LOWER && k0 + 7 < c0) || (A_LOWER && k0 > r0 + 3);
  if (!skip) {
#pragma unroll
    for (int m = k0; m < k0 + 8; m += 4) {
      float4 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (r0 + i) * lda + m);
#pragma unroll
      for (int u = 0; u < 4; ++u) b[u] = *reinterpret_cast<const float4*>(B + (m + u) * ldb + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float av[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc[i][0] = fmaf(av[u], b[u].x, acc[i][0]);
          acc[i][1] = fmaf(av[u], b[u].y, acc[i][1]);
          acc[i][2] = fmaf(av[u], b[u].z, acc[i][2]);
          acc[i][3] = fmaf(av[u], b[u].w, acc[i][3]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(P + (kg * 32 + r0 + i) * 32 + c0) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  named_sync(nb, 256);
  const int r = t >> 3, c = (t & 7) * 4;
  float4 sum = *reinterpret_cast<const float4*>(P + r * 32 + c);
#pragma unroll
  for (int g = 1; g < 4; ++g) {
    const float4 v = *reinterpret_cast<const float4*>(P + (g * 32 + r) * 32 + c);
    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
  }
  *reinterpret_cast<float4*>(C + r * ldc + c) =
      make_float4(alpha * sum.x, alpha * sum.y, alpha * sum.z, alpha * sum.w);
}

}  // namespace chunk
}  // namespace hypic
