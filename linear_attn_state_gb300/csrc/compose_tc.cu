// Compose of gated-delta cached pairs on tcgen05 tensor cores, with the seam
// window of every position fused (youleyou.com HYPIC article: linear-layer
// paragraph, S <- T_C S + S(C|0); seam-window paragraph, the w seam tokens run
// under the full prefix and emit o_t = S_t^T q_t).
//
// One CTA per (request, stream) chain.  Per position j:
//   seam:     the w seam tokens, in chunks of up to 8 (below), o_t per token
//   compose:  S <- c_j Qhat_j S + S_j,  c_j = e^{log_T} 2^{exp2}
// The product is computed transposed, D = S^T Qhat_j^T (M = dv, N = dk, K = dk),
// so that the epilogue thread n owns column n of S.  A = S^T sits in tensor
// memory, B = Qhat_j^T in shared memory, both fp16 split into hi + lo (lo
// scaled by 2^11, after exact power-of-two normalisation of each operand);
// three MMAs (hi*hi, hi*lo + lo*hi) with fp32 accumulators give the product to
// about fp32 accuracy.
//
// Seam chunks.  Unrolling the gated-delta token recurrence over a chunk of n
// tokens from the state S_0 (rows r_s of R are the chunk's effective writes):
//   E[t][s] = prod_{s < u <= t} alpha_u,  gamma_t = prod_{u <= t} alpha_u,
//   (I + strictly_lower(diag(beta) K K^T) o E) R = diag(beta) V - diag(beta gamma) K S_0,
// so with Inv the inverse of the unit lower-triangular matrix on the left,
//   W = Inv diag(beta gamma) K,  U~ = Inv diag(beta) V,  R = U~ - W S_0,
//   o_t = gamma_t S_0^T q_t + sum_{s <= t} E[t][s] (q_t . k_s) r_s,
//   S_n = gamma_{n-1} S_0 + Kbar^T R,   Kbar_s = E[n-1][s] k_s.
// Only the products with S_0 depend on the state.  seam_prep_kernel computes
// the rest for every chunk of every position at once (a chunk record: the rows
// of W and gamma Q as the B operand of one N = 16 MMA, Kbar as the B operand
// of the update, U~ and the small tables), and the chain runs, per chunk:
// A = S_0^T, P = [W ; gamma Q] S_0 on the tensor cores, R on CUDA cores, then
// D_u = R^T Kbar on the tensor cores (A = R^T) while o_t is computed, and
// x <- gamma x + D_u.
//
// When the positions reuse each pair twice or more on average, qop_prep_kernel
// first writes every pair's Qhat once in the B operand format, and the kernel
// (PREP) bulk-copies those images into two B buffers instead of converting.
//
// Warp roles (384 threads): warp 0 MMA issuer, warp 1 producer (the chunk
// records of each position by bulk copy into the record slot, then B_j (PREP)
// or the fp32 Qhat_j tile, and the S_j tile, plus an L2 prefetch one position
// further), warps 2-3 convert Qhat_j into the B operand (idle with PREP;
// without a seam window they take its first kHelpRow rows and the state warps,
// idle then, the rest), warps 4-11 own the state (two threads per column: seam
// chunks, epilogue, A operand) and signal the issuer and producer per warp.
// Tensor memory: [0,128) D hi*hi, [128,256) D cross terms (also D_u of the
// seam update, free until the position's compose), [256,320) A hi, [320,384)
// A lo (fp16 pairs, element k in the low half of column k/2), [384,400) and
// [400,416) the seam product P (hi*hi, cross terms).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "hypic_internal.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kThreads = 384;
constexpr int kH = 64;                 // state rows per state thread (two threads per column)
constexpr uint32_t OFF_QS = 0;        // Qhat_j staging fp32 [128 i][128 k] (64 KB)
constexpr uint32_t OFF_SJ = 65536;    // S_j staging fp32 [128 i][128 n] (64 KB)
constexpr uint32_t OFF_BH = 131072;   // B hi: Qhat rows i, K-major SW128, 2 K blocks (32 KB)
constexpr uint32_t OFF_BL = 163840;   // B lo (32 KB)
static_assert(OFF_BL - OFF_BH == 32768 && OFF_QS + 32768 == 32768, "B planes 32 KB apart");
// seam chunk record (one shared-memory slot): the B operand of P, [W ; gamma Q]
// as two [16 rows][128] fp16 K-major SW128 images (hi, lo; rows 0..7 W, rows
// 8..15 gamma Q, each row scaled by a power of two); the B operand of the
// update, Kbar as two [16 s][128 i] fp16 MN-major SW128 images (rows 8..15
// zero, one power of two for the whole record); U~ [8][128] f32; the tables
// (M [8][8] = E o (Q K^T) f32, gamma [8] f32, the B row exponents [16] i32,
// the Kbar exponent i32)
constexpr int kMaxW = kSeamChunk;
constexpr uint32_t kRecW = 0, kRecKb = 8192, kRecU = 16384, kRecT = 20480;   // slot offsets
constexpr uint32_t kRecBytes = 20992;                                             // slot bytes
// In the record (global memory) the Kbar planes keep only their nonzero half
// (rows s < 8: the image's first 2 KB, with MN atoms 1 KB apart and K groups
// 2 KB apart); the slot's other halves are zeroed once.
constexpr uint32_t kGKh = 8192, kGKl = 10240, kGU = 12288, kGT = 16384;
static_assert(kGT + 512 == kSeamRecordBytes, "seam record size");
constexpr uint32_t OFF_WB = 196608;                 // the record slot (1024-aligned)
constexpr uint32_t SMEM_DYN = OFF_WB + kRecBytes + 1024;
constexpr uint32_t T_DM = 0, T_DC = 128, T_AH = 256, T_AL = 320, T_DS = 384, T_DSC = 400;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdBMN = 1u << 16;  // instruction descriptor: B MN-major
constexpr float kLoScale = 2048.f;     // 2^11
constexpr float kLoUnscale = 1.f / 2048.f;
constexpr uint32_t kDrainLimit = 1u << 20;
constexpr int kHelpRow = 16;           // help mode: the converter warps convert rows 0..15 of B

enum {
  C_QFULL = 0, C_QFREE, C_SFULL, C_SFREE, C_BREADY, C_AREADY, C_DDONE, C_DRAIN,
  C_WFULL, C_WFREE, C_A0READY, C_SDONE, C_URDY, C_UDONE,
  C_BFULL1, C_BEMPTY0, C_BEMPTY1,   // operand copies: B double-buffered (C_BREADY fills buffer 0)
  C_EAREADY,                        // converter: Qhat_j's exponent is known (the state warps help)
  C_COUNT
};

struct CCtl {
  uint64_t bar[C_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t qexp[4];      // power-of-two exponent of max|Qhat_j| (ring by position mod 4)
  uint32_t qmax;        // converter: max |Qhat| bits
  float xmax[2][128];   // state: max |S| of each row half of each column
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// x with the mantissa truncated to 10 stored bits (11 significant): exact in fp16
// whenever x is in fp16's normal range
__device__ __forceinline__ float trunc11(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// 32 lanes x 8 / 4 consecutive columns
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// contiguous global -> shared copy (addresses and size multiples of 16 bytes)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
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
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void l2_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
// D (+)= A[tmem] * B[smem], kind::f16
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
// The 24 MMAs of a split product over K = 128 from one asm block: for each
// K step ks, D_hi (+)= A_hi B_hi and D_cross (+)= A_hi B_lo + A_lo B_hi, with
// A in tensor memory (8 columns a step) and B a K-major SW128 image whose K
// blocks (64 wide) are KB bytes apart and whose lo plane starts LO bytes after
// the hi plane.  Descriptor increments are compile-time immediates.
template <int KB, int LO>
__device__ __forceinline__ void mma24_split(uint32_t dh, uint32_t dx, uint32_t ah, uint32_t al,
                                            uint64_t bh, uint32_t id) {
#define HYPIC_BO(ks) (((ks) >> 2) * (KB / 16) + ((ks) & 3) * 2)
  asm volatile(
      "{\n .reg .pred f, t;\n .reg .b32 ta, tl;\n .reg .b64 yh, yl;\n"
      " setp.ne.b32 f, %6, %6;\n setp.eq.b32 t, %6, %6;\n"
      " add.u32 ta, %2, 0;\n add.u32 tl, %3, 0;\n"
      " add.s64 yh, %4, %7;\n add.s64 yl, %4, %15;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, f;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, f;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 8;\n add.u32 tl, %3, 8;\n"
      " add.s64 yh, %4, %8;\n add.s64 yl, %4, %16;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 16;\n add.u32 tl, %3, 16;\n"
      " add.s64 yh, %4, %9;\n add.s64 yl, %4, %17;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 24;\n add.u32 tl, %3, 24;\n"
      " add.s64 yh, %4, %10;\n add.s64 yl, %4, %18;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 32;\n add.u32 tl, %3, 32;\n"
      " add.s64 yh, %4, %11;\n add.s64 yl, %4, %19;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 40;\n add.u32 tl, %3, 40;\n"
      " add.s64 yh, %4, %12;\n add.s64 yl, %4, %20;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 48;\n add.u32 tl, %3, 48;\n"
      " add.s64 yh, %4, %13;\n add.s64 yl, %4, %21;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      " add.u32 ta, %2, 56;\n add.u32 tl, %3, 56;\n"
      " add.s64 yh, %4, %14;\n add.s64 yl, %4, %22;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yh, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], yl, %5, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%1], [tl], yh, %5, t;\n"
      "}"
      :
      : "r"(dh), "r"(dx), "r"(ah), "r"(al), "l"(bh), "r"(id), "r"(0u),
        "n"(HYPIC_BO(0)), "n"(HYPIC_BO(1)), "n"(HYPIC_BO(2)), "n"(HYPIC_BO(3)),
        "n"(HYPIC_BO(4)), "n"(HYPIC_BO(5)), "n"(HYPIC_BO(6)), "n"(HYPIC_BO(7)),
        "n"(HYPIC_BO(0) + LO / 16), "n"(HYPIC_BO(1) + LO / 16), "n"(HYPIC_BO(2) + LO / 16),
        "n"(HYPIC_BO(3) + LO / 16), "n"(HYPIC_BO(4) + LO / 16), "n"(HYPIC_BO(5) + LO / 16),
        "n"(HYPIC_BO(6) + LO / 16), "n"(HYPIC_BO(7) + LO / 16)
      : "memory");
#undef HYPIC_BO
}

// exponent e with 2^e <= m < 2^(e+1) (m > 0); 0 for m == 0
__device__ __forceinline__ int floor_log2(float m) {
  if (!(m > 0.f)) return 0;
  int e;
  frexpf(m, &e);
  return e - 1;
}

}  // namespace

// Seam chunk records: one warp per (request, position, chunk, stream); lane L
// owns channels 4L .. 4L+3.  Inputs are the chunk's n <= 8 tokens; rows past n
// come out zero, so the chain treats every chunk as 8 tokens.
constexpr int kPrepWarps = 4;
__device__ __forceinline__ float4 ld4g(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4g(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
// Two values x, y times a power of two sc as fp16 pairs: hi = fp16(trunc11(x) sc)
// (exact) and lo = fp16((x - trunc11(x)) sc 2^11); sc2 = (sc, sc), sl2 = sc 2^11.
__device__ __forceinline__ void split_pair(float x, float y, float2 sc2, float2 sl2, uint32_t& hi,
                                           uint32_t& lo) {
  const float2 h = __fmul2_rn(make_float2(trunc11(x), trunc11(y)), sc2);
  const float2 l = __ffma2_rn(make_float2(x, y), sl2, __fmul2_rn(h, make_float2(-2048.f, -2048.f)));
  hi = h2u(__floats2half2_rn(h.x, h.y));
  lo = h2u(__floats2half2_rn(l.x, l.y));
}

// Convert float4 items [first, end) of the staged fp32 Qhat tile (item e: row
// e / 32, k = 4 (e mod 32) .. +3) into the B operand (fp16 hi, lo planes 32 KB
// apart, K-major SW128), by `nt` threads from thread index t.
__device__ __forceinline__ void convert_b_items(const float* qs, uint8_t* bh, int first, int end,
                                                int t, int nt, float sc) {
  const float2 sc2 = make_float2(sc, sc), sl2 = make_float2(sc * kLoScale, sc * kLoScale);
#pragma unroll 4
  for (int e = first + t; e < end; e += nt) {
    const int i = e >> 5, k4 = e & 31;
    const float4 v = reinterpret_cast<const float4*>(qs)[e];
    uint32_t h0, h1, l0, l1;
    split_pair(v.x, v.y, sc2, sl2, h0, l0);
    split_pair(v.z, v.w, sc2, sl2, h1, l1);
    const uint32_t off = sw128_off(i, 4 * k4, 128);
    *reinterpret_cast<uint2*>(bh + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(bh + 32768 + off) = make_uint2(l0, l1);
  }
}

// four values times sc as fp16 hi (11 significant bits, exact) and lo = (a - hi) 2^11
__device__ __forceinline__ void split_h4(const float4& v, float sc, uint2& hi, uint2& lo) {
  const float a0 = v.x * sc, a1 = v.y * sc, a2 = v.z * sc, a3 = v.w * sc;
  const float h0 = trunc11(a0), h1 = trunc11(a1), h2 = trunc11(a2), h3 = trunc11(a3);
  hi = make_uint2(h2u(__floats2half2_rn(h0, h1)), h2u(__floats2half2_rn(h2, h3)));
  lo = make_uint2(h2u(__floats2half2_rn((a0 - h0) * kLoScale, (a1 - h1) * kLoScale)),
                  h2u(__floats2half2_rn((a2 - h2) * kLoScale, (a3 - h3) * kLoScale)));
}
__device__ __forceinline__ float dot4(const float4& a, const float4& b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// Warp reduce-scatter of 32 per-lane values: lane L returns the warp's sum of entry L.
__device__ __forceinline__ float warp_rsum32(float (&a)[32], int lane) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int v = 0; v < m; ++v) {
      const float send = up ? a[v] : a[v + m];
      const float keep = up ? a[v + m] : a[v];
      a[v] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return a[0];
}

template <typename Tin>
__global__ void __launch_bounds__(32 * kPrepWarps, 4)
    seam_prep_kernel(const __grid_constant__ ComposeParams p, int64_t n_rec) {
  __shared__ float scratch[kPrepWarps][512];
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int64_t rec = static_cast<int64_t>(blockIdx.x) * kPrepWarps + wp;
  if (rec >= n_rec) return;   // whole warps only: nothing below synchronises the block
  float* al = scratch[wp];    // [8]
  float* be = al + 8;         // [8]
  float* gam = be + 8;        // [8]
  float* dect = gam + 8;      // [8][8] E[t][s], s <= t < n
  float* dots = dect + 64;    // [64]: 28 pairs k_t.k_s (s < t), then 36 pairs q_t.k_s (s <= t)
  float* inv = dots + 64;     // [8][8]
  float* mq = inv + 64;       // [8][8] E o (Q K^T), zero above the diagonal
  float* cw = mq + 64;        // [8][8] Inv[t][s] beta_s gamma_s
  float* cu = cw + 64;        // [8][8] Inv[t][s] beta_s
  int* rexp = reinterpret_cast<int*>(cu + 64);   // [16]
  const int S = p.n_streams, w = p.w, nch = (w + kMaxW - 1) / kMaxW;
  const int s = static_cast<int>(rec % S);
  const int64_t m = rec / S;                       // (request * n_pos + position) * nch + chunk
  const int c = static_cast<int>(m % nch);
  const int n = min(kMaxW, w - kMaxW * c);         // tokens in this chunk (>= 1)
  const int64_t tok0 = (m / nch) * w + kMaxW * c;  // first token of the chunk
  const Tin* kin = static_cast<const Tin*>(p.k);
  const Tin* qin = static_cast<const Tin*>(p.q);
  const Tin* vin = static_cast<const Tin*>(p.v);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 kr[kMaxW], qr[kMaxW], vr[kMaxW];
#pragma unroll
  for (int t = 0; t < kMaxW; ++t) {
    kr[t] = qr[t] = vr[t] = z4;
    if (t < n) {
      const int64_t e = ((tok0 + t) * S + s) * kD + 4 * lane;
      kr[t] = ld4g(kin + e);
      qr[t] = ld4g(qin + e);
      vr[t] = ld4g(vin + e);
    }
  }
  if (lane < kMaxW) {
    const int64_t e = (tok0 + lane) * S + s;
    al[lane] = (lane < n) ? expf(p.log_alpha[e]) : 1.f;
    be[lane] = (lane < n) ? p.beta[e] : 0.f;
  }
  // the 64 dot products -- 28 pairs k_t.k_s (s < t), then 36 pairs q_t.k_s
  // (s <= t), row by row -- in two reduce-scatters of 32
#pragma unroll
  for (int base = 0; base < 64; base += 32) {
    float a[32];
    int pi = 0;   // pair index (a compile-time constant in the unrolled loops)
#pragma unroll
    for (int t1 = 1; t1 < kMaxW; ++t1)
#pragma unroll
      for (int s1 = 0; s1 < t1; ++s1, ++pi)
        if (pi >= base && pi < base + 32) a[pi - base] = dot4(kr[t1], kr[s1]);
#pragma unroll
    for (int t1 = 0; t1 < kMaxW; ++t1)
#pragma unroll
      for (int s1 = 0; s1 <= t1; ++s1, ++pi)
        if (pi >= base && pi < base + 32) a[pi - base] = dot4(qr[t1], kr[s1]);
    dots[base + lane] = warp_rsum32(a, lane);
  }
  __syncwarp();
  // decay tables: E[t][s] (two entries a lane), gamma_t (lanes 0..7)
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int e = lane + 32 * r2, t1 = e >> 3, s1 = e & 7;
    float d = 0.f;
    if (s1 <= t1 && t1 < n) {
      d = 1.f;
      for (int u = s1 + 1; u <= t1; ++u) d *= al[u];
    }
    dect[e] = d;
  }
  if (lane < kMaxW) {
    float d = 0.f;
    if (lane < n) {
      d = 1.f;
      for (int u = 0; u <= lane; ++u) d *= al[u];
    }
    gam[lane] = d;
  }
  __syncwarp();
  // Inv by columns (lanes 0..7: forward substitution on the unit lower-
  // triangular matrix); M = E o (Q K^T) (all lanes, two entries each)
  if (lane < kMaxW) {
    const int jc = lane;
    float xs[kMaxW];
#pragma unroll
    for (int t1 = 0; t1 < kMaxW; ++t1) xs[t1] = (t1 == jc) ? 1.f : 0.f;
#pragma unroll
    for (int t1 = 1; t1 < kMaxW; ++t1) {
      if (t1 > jc && t1 < n) {
        float acc = 0.f;
#pragma unroll
        for (int s1 = 0; s1 < t1; ++s1)
          if (s1 >= jc) acc = fmaf(dots[t1 * (t1 - 1) / 2 + s1] * dect[t1 * 8 + s1], xs[s1], acc);
        xs[t1] = -be[t1] * acc;
      }
    }
#pragma unroll
    for (int t1 = 0; t1 < kMaxW; ++t1) inv[t1 * 8 + jc] = (t1 < n && jc < n) ? xs[t1] : 0.f;
  }
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int e = lane + 32 * r2, t1 = e >> 3, s1 = e & 7;
    mq[e] = (s1 <= t1) ? dots[28 + t1 * (t1 + 1) / 2 + s1] * dect[e] : 0.f;
  }
  __syncwarp();
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int e = lane + 32 * r2, s1 = e & 7;
    cw[e] = inv[e] * be[s1] * gam[s1];
    cu[e] = inv[e] * be[s1];
  }
  __syncwarp();
  // this lane's four channels of the rows of U~ (stored), of gamma Q and W
  // (kept for the P images) and of Kbar (its image); in this order the inputs
  // die early
  uint8_t* out = p.seam_rec + rec * static_cast<int64_t>(kSeamRecordBytes);
  float* uo = reinterpret_cast<float*>(out + kGU);
#pragma unroll
  for (int t1 = 0; t1 < kMaxW; ++t1) {
    float4 uv = z4;
#pragma unroll
    for (int s1 = 0; s1 < kMaxW; ++s1) {
      const float b = cu[t1 * 8 + s1];
      uv.x = fmaf(b, vr[s1].x, uv.x); uv.y = fmaf(b, vr[s1].y, uv.y);
      uv.z = fmaf(b, vr[s1].z, uv.z); uv.w = fmaf(b, vr[s1].w, uv.w);
    }
    *reinterpret_cast<float4*>(uo + t1 * kD + 4 * lane) = uv;
  }
  float4 row[16];
#pragma unroll
  for (int t1 = 0; t1 < kMaxW; ++t1) {
    const float g = gam[t1];
    row[8 + t1] = make_float4(g * qr[t1].x, g * qr[t1].y, g * qr[t1].z, g * qr[t1].w);
  }
#pragma unroll
  for (int t1 = 0; t1 < kMaxW; ++t1) {
    float4 wv = z4;
#pragma unroll
    for (int s1 = 0; s1 < kMaxW; ++s1) {
      const float a = cw[t1 * 8 + s1];
      wv.x = fmaf(a, kr[s1].x, wv.x); wv.y = fmaf(a, kr[s1].y, wv.y);
      wv.z = fmaf(a, kr[s1].z, wv.z); wv.w = fmaf(a, kr[s1].w, wv.w);
    }
    row[t1] = wv;
  }
  {
    // Kbar_s = E[n-1][s] k_s as the update's B operand: element (s, i) of an
    // MN-major [16 s][128 i] image (two 64-wide MN atoms 2 KB apart), one
    // power-of-two scale for the record, fp16 hi + lo
    const float* kb = dect + (n - 1) * 8;
    float mx = 0.f;
#pragma unroll
    for (int t1 = 0; t1 < kMaxW; ++t1) {
      const float f = kb[t1];
      kr[t1] = make_float4(f * kr[t1].x, f * kr[t1].y, f * kr[t1].z, f * kr[t1].w);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(kr[t1].x), fabsf(kr[t1].y)),
                           fmaxf(fabsf(kr[t1].z), fabsf(kr[t1].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int ek = floor_log2(mx);
    const float sc = ldexpf(1.f, -ek);
#pragma unroll
    for (int t1 = 0; t1 < kMaxW; ++t1) {
      uint2 hi, lo;
      split_h4(kr[t1], sc, hi, lo);
      // element (s, i): MN atom i / 64 (1 KB apart), K row s, 16-byte chunk
      // (i / 8) mod 8 swizzled by s
      const uint32_t off = (lane >> 4) * 1024u + t1 * 128u + ((((lane >> 1) & 7) ^ t1) << 4) +
                           (lane & 1) * 8u;
      *reinterpret_cast<uint2*>(out + kGKh + off) = hi;
      *reinterpret_cast<uint2*>(out + kGKl + off) = lo;
    }
    if (lane == 0) reinterpret_cast<int*>(out + kGT)[88] = ek;
  }
  // power-of-two exponent of each B row (max |.| over the 128 channels):
  // reduce-scatter of the 16 maxima over each half warp, then across halves
  {
    float a[16];
#pragma unroll
    for (int t1 = 0; t1 < 16; ++t1)
      a[t1] = fmaxf(fmaxf(fabsf(row[t1].x), fabsf(row[t1].y)),
                    fmaxf(fabsf(row[t1].z), fabsf(row[t1].w)));
#pragma unroll
    for (int mm = 8; mm > 0; mm >>= 1) {
      const bool up = (lane & mm) != 0;
#pragma unroll
      for (int v = 0; v < mm; ++v) {
        const float send = up ? a[v] : a[v + mm];
        const float keep = up ? a[v + mm] : a[v];
        a[v] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, mm));
      }
    }
    const float mx = fmaxf(a[0], __shfl_xor_sync(0xffffffffu, a[0], 16));   // row lane & 15
    if (lane < 16) rexp[lane] = floor_log2(mx);
  }
  __syncwarp();
  // P images: (row, channels 4L..4L+3) at the K-major SW128 offset
#pragma unroll
  for (int t1 = 0; t1 < 16; ++t1) {
    uint2 hi, lo;
    split_h4(row[t1], ldexpf(1.f, -rexp[t1]), hi, lo);
    const uint32_t off = sw128_off(t1, 4 * lane, 16);
    *reinterpret_cast<uint2*>(out + kRecW + off) = hi;
    *reinterpret_cast<uint2*>(out + kRecW + 4096 + off) = lo;
  }
  // tables: M [64], gamma [8], the P row exponents [16] (the Kbar exponent at 88)
  float* tab = reinterpret_cast<float*>(out + kGT);
  tab[lane] = mq[lane];
  tab[32 + lane] = mq[32 + lane];
  if (lane < 8) tab[64 + lane] = gam[lane];
  if (lane < 16) reinterpret_cast<int*>(tab)[72 + lane] = rexp[lane];
}

// Operand copy of each pair's Qhat, for composes that reuse pairs: one CTA of
// 256 threads per (segment, stream) unit writes the B images (fp16 hi and lo
// planes, K-major SW128, exactly the shared-memory layout the compose MMAs
// read) after normalising by the power of two of max |Qhat|, and that exponent.
// The arithmetic is the in-kernel converter's, so both paths give the same bits.
__global__ void __launch_bounds__(256) qop_prep_kernel(const float* __restrict__ Qhat,
                                                       uint8_t* __restrict__ qop,
                                                       int32_t* __restrict__ qexp) {
  __shared__ float wmax[8];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t u = blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(Qhat + u * kD * kD);
  float4 v[16];
  float m = 0.f;
#pragma unroll
  for (int r2 = 0; r2 < 16; ++r2) {
    v[r2] = src[tid + 256 * r2];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[r2].x), fabsf(v[r2].y)), fmaxf(fabsf(v[r2].z), fabsf(v[r2].w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[tid >> 5] = m;
  __syncthreads();
  m = wmax[0];
#pragma unroll
  for (int w2 = 1; w2 < 8; ++w2) m = fmaxf(m, wmax[w2]);
  const int ea = floor_log2(m);
  const float sc = ldexpf(1.f, -ea);
  uint8_t* dst = qop + u * static_cast<int64_t>(kQopBytes);
#pragma unroll
  for (int r2 = 0; r2 < 16; ++r2) {
    const int e = tid + 256 * r2, i = e >> 5, k4 = e & 31;   // row i, k = 4 k4 .. 4 k4 + 3
    uint2 hi, lo;
    split_h4(v[r2], sc, hi, lo);
    const uint32_t off = sw128_off(i, 4 * k4, 128);
    *reinterpret_cast<uint2*>(dst + off) = hi;
    *reinterpret_cast<uint2*>(dst + 32768 + off) = lo;
  }
  if (tid == 0) qexp[u] = ea;
}

template <bool PREP>
__global__ void __launch_bounds__(kThreads, 1)
    compose_tc_kernel(const __grid_constant__ ComposeParams p,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_s) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ CCtl ctl;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chain = blockIdx.x;
  const int r = chain / p.n_streams, s = chain % p.n_streams;
  const int S = p.n_streams;
  const int P = p.n_pos;
  const int nch = (p.w + kMaxW - 1) / kMaxW;   // seam chunks per position
  // Without a seam window and without operand copies the state warps are idle
  // while the converter works: they convert rows kHelpRow.. of each B.
  const bool help = !PREP && p.w == 0;
  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    // the state role signals per warp: 8 arrivals (URDY: the 4 warps of row half 0)
    for (int i = 0; i < C_COUNT; ++i)
      mbar_init(BAR(i), (i == C_A0READY || i == C_AREADY || i == C_SFREE || i == C_WFREE) ? 8
                        : (i == C_URDY)                                                 ? 4
                        : (help && (i == C_QFREE || i == C_BREADY))                     ? 2
                                                                                        : 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_s);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t limit = p.spin_limit;
  auto wait_k = [&](int i, uint32_t k) -> bool {
    const uint32_t b = BAR(i), par = k & 1u;
    if (warp == 0) {
      // the MMA issuer polls without suspending, so it issues as soon as an
      // input lands (64 polls a round; the limit counts rounds)
      for (uint32_t n = 0; n < limit; ++n) {
        for (int u = 0; u < 64; ++u)
          if (mbar_test(b, par)) return true;
        if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
      }
    } else {
      for (uint32_t n = 0; n < limit; ++n) {
        if (mbar_try(b, par)) return true;
        if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
      }
    }
    if (atomicExch(&ctl.abort_flag, 1) == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, 200 + i);
    return false;
  };
  // segment of position j, or -1 when out of range (that position is skipped);
  // the chain roles load the entry a position ahead and check it on use
  auto order_at = [&](int j) -> int { return p.order[static_cast<int64_t>(r) * P + j]; };
  auto seg_ok = [&](int sg) -> int { return (sg >= 0 && sg < p.n_seg) ? sg : -1; };
  auto seg_at = [&](int j) -> int { return seg_ok(order_at(j)); };

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      int sg_next = P > 0 ? order_at(0) : -1;   // the order entry one position ahead
      for (int j = 0; j < P && ok; ++j) {
        const int sg = seg_ok(sg_next);
        if (j + 1 < P) sg_next = order_at(j + 1);
        // seam chunks: P = [W ; gamma Q] S_0 into the seam tiles (hi*hi, cross
        // terms); then the update D_u = R^T Kbar into the compose accumulators
        // (free until this position's compose)
        for (int c = 0; c < nch && ok; ++c) {
          const uint32_t q = static_cast<uint32_t>(j * nch + c);
          if (!(ok = wait_k(C_WFULL, q) && wait_k(C_A0READY, q))) break;
          tc_fence_after();
          mma24_split<2048, 4096>(tmem + T_DS, tmem + T_DSC, tmem + T_AH, tmem + T_AL,
                                  desc_sw128(sb + OFF_WB + kRecW), idesc_f16(128, 16));
          mma_commit(BAR(C_SDONE));
          if (!(ok = wait_k(C_URDY, q))) break;
          tc_fence_after();
          const uint32_t iu = idesc_f16(128, 128) | kIdBMN;
          // Kbar image: MN atoms 1 KB apart, 8-row K groups 2 KB apart
          const uint64_t kh = desc_mn(sb + OFF_WB + kRecKb, 1024, 2048),
                         kl = desc_mn(sb + OFF_WB + kRecKb + 4096, 1024, 2048);
          mma_ts(tmem + T_DM, tmem + T_AH, kh, iu, 0);
          mma_ts(tmem + T_DC, tmem + T_AH, kl, iu, 0);
          mma_ts(tmem + T_DC, tmem + T_AL, kh, iu, 1);
          mma_commit(BAR(C_UDONE));
        }
        if (!ok) break;
        // B_j: the converter's buffer, or operand copy j in buffer j mod 2
        const uint32_t bb = PREP ? (static_cast<uint32_t>(j) & 1u) : 0u;
        const bool bf = PREP ? wait_k(bb ? C_BFULL1 : C_BREADY, j >> 1) : wait_k(C_BREADY, j);
        if (!(ok = wait_k(C_AREADY, j) && bf)) break;
        tc_fence_after();
        if (sg >= 0) {
          mma24_split<16384, 32768>(tmem + T_DM, tmem + T_DC, tmem + T_AH, tmem + T_AL,
                                    desc_sw128(sb + (bb ? OFF_QS : OFF_BH)), idesc_f16(128, 128));
        }
        mma_commit(BAR(C_DDONE));
        if (PREP) mma_commit(BAR(bb ? C_BEMPTY1 : C_BEMPTY0));
      }
      if (!ok) {
        mma_commit(BAR(C_DRAIN));
        mbar_wait(BAR(C_DRAIN), 0, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- producer
    // per position j: its seam chunk records into the record slot (once the
    // state role has released the previous record), then Qhat_j and S_j
    bool ok = true;
    uint32_t qiss = 0, siss = 0, wiss = 0, biss0 = 0, biss1 = 0;
    for (int j = 0; j < P && ok; ++j) {
      const int sg = seg_at(j);
      if (lane == 0) {
        for (int c = 0; c < nch && ok; ++c) {
          const uint32_t q = static_cast<uint32_t>(j * nch + c);
          if (q >= 1 && !wait_k(C_WFREE, q - 1)) {
            ok = false;
            break;
          }
          const uint8_t* src =
              p.seam_rec +
              (((static_cast<int64_t>(r) * P + j) * nch + c) * S + s) *
                  static_cast<int64_t>(kSeamRecordBytes);
          mbar_expect_tx(BAR(C_WFULL), static_cast<uint32_t>(kSeamRecordBytes));
          bulk_load(sb + OFF_WB + kRecW, src, kGKh, BAR(C_WFULL));
          bulk_load(sb + OFF_WB + kRecKb, src + kGKh, 2048, BAR(C_WFULL));
          bulk_load(sb + OFF_WB + kRecKb + 4096, src + kGKl, 2048, BAR(C_WFULL));
          bulk_load(sb + OFF_WB + kRecU, src + kGU, kSeamRecordBytes - kGU, BAR(C_WFULL));
          ++wiss;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        if (j + 1 < P) {  // next position's tiles towards L2
          const int sn = seg_at(j + 1);
          if (sn >= 0) {
            const int32_t row = (sn * S + s) * kD;
            if (!PREP) l2_prefetch_2d(&tm_q, 0, row);
            l2_prefetch_2d(&tm_s, 0, row);
          }
        }
        if (PREP) {
          // operand copy j into B buffer j mod 2, once the MMA two positions back is done
          const uint32_t bb = static_cast<uint32_t>(j) & 1u;
          if (j >= 2 && !wait_k(bb ? C_BEMPTY1 : C_BEMPTY0, (j >> 1) - 1)) {
            ok = false;
          } else {
            const uint32_t bar = BAR(bb ? C_BFULL1 : C_BREADY);
            if (sg >= 0) {
              mbar_expect_tx(bar, static_cast<uint32_t>(kQopBytes));
              bulk_load(sb + (bb ? OFF_QS : OFF_BH),
                        p.qop + (static_cast<int64_t>(sg) * S + s) * static_cast<int64_t>(kQopBytes),
                        static_cast<uint32_t>(kQopBytes), bar);
            } else {
              mbar_arrive(bar);
            }
            if (bb) ++biss1; else ++biss0;
          }
        } else if (j >= 1 && !wait_k(C_QFREE, j - 1)) {
          ok = false;
        } else {
          if (sg >= 0) {
            mbar_expect_tx(BAR(C_QFULL), kD * kD * 4);
            tma_load_2d(sb + OFF_QS, &tm_q, BAR(C_QFULL), 0, (sg * S + s) * kD);
          } else {
            mbar_arrive(BAR(C_QFULL));
          }
          ++qiss;
        }
        if (ok) {
          if (j >= 1 && !wait_k(C_SFREE, j - 1)) {
            ok = false;
          } else {
            if (sg >= 0) {
              mbar_expect_tx(BAR(C_SFULL), kD * kD * 4);
              tma_load_2d(sb + OFF_SJ, &tm_s, BAR(C_SFULL), 0, (sg * S + s) * kD);
            } else {
              mbar_arrive(BAR(C_SFULL));
            }
            ++siss;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0) {
      // drain the copies this thread issued
      if (qiss) mbar_wait(BAR(C_QFULL), (qiss - 1) & 1u, kDrainLimit);
      if (siss) mbar_wait(BAR(C_SFULL), (siss - 1) & 1u, kDrainLimit);
      if (wiss) mbar_wait(BAR(C_WFULL), (wiss - 1) & 1u, kDrainLimit);
      if (biss0) mbar_wait(BAR(C_BREADY), (biss0 - 1) & 1u, kDrainLimit);
      if (biss1) mbar_wait(BAR(C_BFULL1), (biss1 - 1) & 1u, kDrainLimit);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- converter
    // (idle when the operand copies are loaded directly)
    const int ct = tid - 64;  // 0..63
    bool ok = !PREP;
    for (int j = 0; j < P && ok; ++j) {
      const int sg = seg_at(j);
      bool fail = (ct == 0) && !wait_k(C_QFULL, j);
      if (named_or(1, 64, fail)) { ok = false; break; }
      const float* qs = reinterpret_cast<const float*>(sm + OFF_QS);
      int ea = 0;
      if (sg >= 0) {
        float m = 0.f;
#pragma unroll 8
        for (int e = ct; e < 4096; e += 64) {
          const float4 v = reinterpret_cast<const float4*>(qs)[e];
          m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (ct == 0) ctl.qmax = 0u;
        named_sync(1, 64);
        if (lane == 0) atomicMax(&ctl.qmax, __float_as_uint(m));
        named_sync(1, 64);
        ea = floor_log2(__uint_as_float(ctl.qmax));
      }
      if (ct == 0) {
        ctl.qexp[j & 3] = ea;
        if (help) mbar_arrive(BAR(C_EAREADY));
      }
      // B is free once the previous position's MMAs are done
      fail = (ct == 0) && j >= 1 && !wait_k(C_DDONE, j - 1);
      if (named_or(1, 64, fail)) { ok = false; break; }
      if (sg >= 0 && help) {
        convert_b_items(qs, sm + OFF_BH, 0, 32 * kHelpRow, ct, 64, ldexpf(1.f, -ea));
      } else if (sg >= 0) {
        // thread ct converts k = 4 k4 .. 4 k4 + 3 (k4 = ct mod 32) of rows
        // i = ct / 32 + 2 it: over four consecutive it the swizzle phase i mod 8
        // takes four values, so their offsets are fixed and rows advance by 8
        const float sc = ldexpf(1.f, -ea);
        const float2 sc2 = make_float2(sc, sc), sl2 = make_float2(sc * kLoScale, sc * kLoScale);
        const int k4 = ct & 31, i0 = ct >> 5;
        uint32_t base[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t r7 = static_cast<uint32_t>(i0 + 2 * u);
          base[u] = (k4 >> 4) * 16384u + r7 * 128u + ((((k4 & 15) >> 1) ^ r7) << 4) + (k4 & 1) * 8u;
        }
        const float4* q4 = reinterpret_cast<const float4*>(qs) + ct;
#pragma unroll 2
        for (int mrow = 0; mrow < 16; ++mrow) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float4 v = q4[256 * mrow + 64 * u];
            uint32_t h0, h1, l0, l1;
            split_pair(v.x, v.y, sc2, sl2, h0, l0);
            split_pair(v.z, v.w, sc2, sl2, h1, l1);
            const uint32_t off = base[u] + 1024u * mrow;
            *reinterpret_cast<uint2*>(sm + OFF_BH + off) = make_uint2(h0, h1);
            *reinterpret_cast<uint2*>(sm + OFF_BL + off) = make_uint2(l0, l1);
          }
        }
      }
      fence_proxy_async();
      named_sync(1, 64);
      if (ct == 0) {
        mbar_arrive(BAR(C_QFREE));
        mbar_arrive(BAR(C_BREADY));
      }
    }
  } else {
    // ---------------------------------------------------------------- state owners
    // Two threads per column n of S (warps 4-7 rows 0..63, warps 8-11 rows
    // 64..127; TMEM lane = n).  Per seam chunk: A = S_0^T, P from the tensor
    // cores, R, then the update D_u = R^T Kbar on the tensor cores while the
    // chunk's outputs are computed, and x <- gamma x + D_u; per position:
    // A = S_w^T (and, without a seam window, rows of B) and the compose
    // epilogue.
    const int n = (warp & 3) * 32 + lane;        // column n of S = TMEM lane
    const int h = (warp - 4) >> 2;               // row half
    const int i0 = 64 * h;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int et = tid - 128;                     // 0..255
    const int64_t st_base = (static_cast<int64_t>(r) * S + s) * kD * kD;
    float x[kH];
#pragma unroll
    for (int i = 0; i < kH; ++i) x[i] = p.state_in ? p.state_in[st_base + (i0 + i) * kD + n] : 0.f;
    if (p.w > 0) {
      // rows 8..15 of the Kbar planes in the record slot are zero, never copied
      const uint32_t z = OFF_WB + kRecKb + 2048 + (et >> 7) * 4096 + (et & 127) * 16;
      *reinterpret_cast<uint4*>(sm + z) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async();   // read by the tensor core
    }
    // A operand: S^T row n, columns (k) i0..i0+63 of this half, normalised by
    // 2^-eb with eb from this column's max |S| (the two row halves exchange
    // their maxima; a row scale of A scales the same row of every product),
    // fp16 hi + lo; returns eb
    auto write_A = [&]() -> int {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < kH; ++i) m = fmaxf(m, fabsf(x[i]));
      ctl.xmax[h][n] = m;
      named_sync(2, 256);
      const int eb = floor_log2(fmaxf(m, ctl.xmax[h ^ 1][n]));
      const float sc = ldexpf(1.f, -eb);
      const float2 sc2 = make_float2(sc, sc), sl2 = make_float2(sc * kLoScale, sc * kLoScale);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          split_pair(x[16 * bb + 2 * e], x[16 * bb + 2 * e + 1], sc2, sl2, hi[e], lo[e]);
        const uint32_t col = (i0 >> 1) + 8 * bb;
        tmem_st8(tmem + lane_off + T_AH + col, hi);
        tmem_st8(tmem + lane_off + T_AL + col, lo);
      }
      tmem_wait_st();
      return eb;
    };
    bool ok = true;
    // the next position's order entry and pair scalars, loaded while the chain
    // waits on the tensor cores of the current one
    int sg_nx = -1, raw_nx = -1, x2_nx = 0, qe_nx = 0;
    float lt_nx = 0.f;
    auto prefetch = [&](int jn) {
      sg_nx = seg_ok(raw_nx);
      if (sg_nx >= 0) {
        const int64_t u = static_cast<int64_t>(sg_nx) * S + s;
        lt_nx = p.log_T[u];
        x2_nx = p.exp2[u];
        if (PREP) qe_nx = p.qop_exp[u];
      }
      raw_nx = (jn + 1 < P) ? order_at(jn + 1) : -1;
    };
    if (P > 0) {
      raw_nx = order_at(0);
      prefetch(0);
    }
    for (int j = 0; j < P && ok; ++j) {
      const int sg = sg_nx;
      const float lt = lt_nx;
      const int x2 = x2_nx, qe = qe_nx;
      if (sg < 0 && et == 0) report(p.ws, HYPIC_ERR_INDEX, 210);
      // ---- seam chunks of position j
      for (int c = 0; c < nch && ok; ++c) {
        const uint32_t q = static_cast<uint32_t>(j * nch + c);
        const int nt = min(kMaxW, p.w - kMaxW * c);                 // tokens in the chunk
        const int64_t tok0 = (static_cast<int64_t>(r) * P + j) * p.w + kMaxW * c;
        const float* wu = reinterpret_cast<const float*>(sm + OFF_WB + kRecU);
        const float* mq = reinterpret_cast<const float*>(sm + OFF_WB + kRecT);
        const float* gam = mq + 64;
        const int* rexp = reinterpret_cast<const int*>(mq + 72);
        // A = S_0^T; A is free: the previous chunk's product and the previous
        // position's compose were waited for before x was last written
        const int eb0 = write_A();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C_A0READY));
        bool sf = (et == 0) && !(wait_k(C_SDONE, q) && wait_k(C_WFULL, q));   // (record landed)
        if (named_or(2, 256, sf)) { ok = false; break; }
        tc_fence_after();
        // P[t][n] = D 2^(eb0 + rexp[t]), the scale an exact power of two built
        // from the exponent: rows 0..7 (W S_0) and this row half's four rows of
        // gamma Q S_0 (tokens 4h .. 4h+3)
        uint32_t dw[8], cw[8], dq[4], cq[4];
        tmem_ld8(tmem + lane_off + T_DS, dw);
        tmem_ld8(tmem + lane_off + T_DSC, cw);
        tmem_ld4(tmem + lane_off + T_DS + 8 + 4 * h, dq);
        tmem_ld4(tmem + lane_off + T_DSC + 8 + 4 * h, cq);
        tmem_wait_ld();
        auto pscale = [&](int row) {
          const int e = min(max(eb0 + rexp[row], -126), 127);
          return __int_as_float((e + 127) << 23);
        };
        // R (rows past the chunk are zero: U~ and P vanish there)
        float rv[kMaxW];
#pragma unroll
        for (int t1 = 0; t1 < kMaxW; ++t1)
          rv[t1] = wu[t1 * kD + n] -
                   (__uint_as_float(dw[t1]) + __uint_as_float(cw[t1]) * kLoUnscale) * pscale(t1);
        // S_n = gamma_{n-1} S_0 + Kbar^T R, the product on the tensor cores:
        // A = R^T (row n, K = s, s >= 8 zero) scaled by 2^-er from this
        // column's R, fp16 hi + lo, written by row half 0 over the A tiles
        // (S_0^T is no longer needed); D_u lands in the compose accumulators
        int er;
        {
          float mr = 0.f;
#pragma unroll
          for (int t1 = 0; t1 < kMaxW; ++t1) mr = fmaxf(mr, fabsf(rv[t1]));
          er = floor_log2(mr);
        }
        if (h == 0) {
          const float sc = ldexpf(1.f, -er);
          const float2 sc2 = make_float2(sc, sc), sl2 = make_float2(sc * kLoScale, sc * kLoScale);
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            split_pair(rv[2 * e], rv[2 * e + 1], sc2, sl2, hi[e], lo[e]);
            hi[4 + e] = lo[4 + e] = 0u;
          }
          tmem_st8(tmem + lane_off + T_AH, hi);
          tmem_st8(tmem + lane_off + T_AL, lo);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C_URDY));
        }
        // outputs (while the update runs): tokens 0..3 by row half 0, 4..7 by
        // row half 1 (M is zero above the diagonal and past the chunk)
        {
          float ov[4];
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const int t1 = 4 * h + tt;
            float o = (__uint_as_float(dq[tt]) + __uint_as_float(cq[tt]) * kLoUnscale) * pscale(8 + t1);
            const float4 m0 = *reinterpret_cast<const float4*>(mq + t1 * 8);
            const float4 m1 = *reinterpret_cast<const float4*>(mq + t1 * 8 + 4);
            o = fmaf(m0.x, rv[0], o); o = fmaf(m0.y, rv[1], o);
            o = fmaf(m0.z, rv[2], o); o = fmaf(m0.w, rv[3], o);
            o = fmaf(m1.x, rv[4], o); o = fmaf(m1.y, rv[5], o);
            o = fmaf(m1.z, rv[6], o); o = fmaf(m1.w, rv[7], o);
            ov[tt] = o;
          }
          const int64_t ob = ((tok0 + 4 * h) * S + s) * kD + n, ostep = static_cast<int64_t>(S) * kD;
          const int nv = min(4, nt - 4 * h);   // this half's tokens inside the chunk
          if (p.o_bf16) {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out_o) + ob;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt)
              if (tt < nv) o[tt * ostep] = __float2bfloat16_rn(ov[tt]);
          } else {
            float* o = static_cast<float*>(p.out_o) + ob;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt)
              if (tt < nv) o[tt * ostep] = ov[tt];
          }
        }
        bool uf = (et == 0) && !wait_k(C_UDONE, q);
        if (named_or(2, 256, uf)) { ok = false; break; }
        tc_fence_after();
        {
          const float gw = gam[nt - 1];
          const int eu = min(max(er + reinterpret_cast<const int*>(mq)[88], -126), 127);
          const float us = __int_as_float((eu + 127) << 23);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            uint32_t dm[16], dc[16];
            tmem_ld16(tmem + lane_off + T_DM + i0 + 16 * bb, dm);
            tmem_ld16(tmem + lane_off + T_DC + i0 + 16 * bb, dc);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int i = 16 * bb + e;
              const float d = __uint_as_float(dm[e]) + __uint_as_float(dc[e]) * kLoUnscale;
              x[i] = fmaf(gw, x[i], us * d);
            }
          }
        }
        tc_fence_before();
        __syncwarp();   // this warp has read the record slot and the seam tiles
        if (lane == 0) mbar_arrive(BAR(C_WFREE));
      }
      if (!ok) break;
      // ---- A operand S_w^T for the compose
      int eb = 0;
      if (sg >= 0) eb = write_A();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C_AREADY));
      if (j + 1 < P) prefetch(j + 1);
      if (help) {
        // rows kHelpRow.. of B_j (B is free: MMA j-1 was waited for before x)
        bool hf = (et == 0) && !(wait_k(C_QFULL, j) && wait_k(C_EAREADY, j));
        if (named_or(2, 256, hf)) { ok = false; break; }
        if (sg >= 0)
          convert_b_items(reinterpret_cast<const float*>(sm + OFF_QS), sm + OFF_BH, 32 * kHelpRow,
                          4096, et, 256, ldexpf(1.f, -ctl.qexp[j & 3]));
        fence_proxy_async();
        named_sync(2, 256);
        if (et == 0) {
          mbar_arrive(BAR(C_QFREE));
          mbar_arrive(BAR(C_BREADY));
        }
      }
      // ---- epilogue: x <- c * D + S_j (column n, this row half)
      bool fail = (et == 0) && !(wait_k(C_DDONE, j) && wait_k(C_SFULL, j));
      if (named_or(2, 256, fail)) { ok = false; break; }
      tc_fence_after();
      if (sg >= 0) {
        const int ea = PREP ? qe : ctl.qexp[j & 3];
        const float c = expf(lt + static_cast<float>(x2 + ea + eb) * 0.69314718055994531f);
        const float* sj = reinterpret_cast<const float*>(sm + OFF_SJ);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          uint32_t dm[16], dc[16];
          tmem_ld16(tmem + lane_off + T_DM + i0 + 16 * bb, dm);
          tmem_ld16(tmem + lane_off + T_DC + i0 + 16 * bb, dc);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 16 * bb + e;
            const float d = __uint_as_float(dm[e]) + __uint_as_float(dc[e]) * kLoUnscale;
            x[i] = fmaf(c, d, sj[(i0 + i) * kD + n]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C_SFREE));
    }
    if (ok) {
      float* out = p.state_out + st_base;
#pragma unroll
      for (int i = 0; i < kH; ++i) out[(i0 + i) * kD + n] = x[i];
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_c() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D map over n_units x 128 rows of 128 fp32 (one 64 KB tile per unit)
bool make_map_f32(CUtensorMap* m, const float* base, int64_t n_units) {
  auto fn = encode_fn_c();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(n_units * kD)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kD)};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool compose_tc_supported(const ComposeParams& p) {
  // seam windows of any length run as chunks of up to 8 tokens (the chunk
  // records live in the workspace, sized by hypic_compose_workspace_bytes)
  const int64_t n_seam_tok = static_cast<int64_t>(p.n_req) * p.n_pos * p.w;
  return p.kind == HYPIC_GDN && (p.w == 0 || (p.seam_kind == HYPIC_GDN && p.seam_rec)) &&
         p.dk == kD && p.dv == kD && p.n_seg > 0 && n_seam_tok < (int64_t{1} << 31);
}

cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t st) {
  const int64_t n_units = static_cast<int64_t>(p.n_seg) * p.n_streams;
  CUtensorMap mq, ms;
  if (!make_map_f32(&mq, p.Qhat, n_units) || !make_map_f32(&ms, p.Sc, n_units))
    return cudaErrorInvalidValue;
  if (p.w > 0) {
    const int64_t n_rec = static_cast<int64_t>(p.n_req) * p.n_pos * ((p.w + kMaxW - 1) / kMaxW) *
                          p.n_streams;
    if (n_rec > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>((n_rec + kPrepWarps - 1) / kPrepWarps);
    if (p.seam_dtype == HYPIC_F32)
      seam_prep_kernel<float><<<grid, 32 * kPrepWarps, 0, st>>>(p, n_rec);
    else
      seam_prep_kernel<__nv_bfloat16><<<grid, 32 * kPrepWarps, 0, st>>>(p, n_rec);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const bool prep = p.qop != nullptr;
  if (prep) {
    if (n_units > 0x7FFFFFFF) return cudaErrorInvalidValue;
    qop_prep_kernel<<<static_cast<unsigned>(n_units), 256, 0, st>>>(p.Qhat, p.qop, p.qop_exp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kern = prep ? compose_tc_kernel<true> : compose_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  kern<<<p.n_req * p.n_streams, kThreads, SMEM_DYN, st>>>(p, mq, ms);
  return cudaGetLastError();
}

}  // namespace hypic
