// Compose of gated-delta cached pairs on tcgen05 tensor cores, with the seam
// window of every position fused (youleyou.com HYPIC article: linear-layer
// paragraph, S <- T_C S + S(C|0); seam-window paragraph, the w seam tokens run
// under the full prefix and emit o_t = S_t^T q_t).
//
// One CTA per (request, stream) chain.  Per position j:
//   seam:     w rank-1 token updates of the state, o_t per token (fp32)
//   compose:  S <- c_j Qhat_j S + S_j,  c_j = e^{log_T} 2^{exp2}
// The product is computed transposed, D = S^T Qhat_j^T (M = dv, N = dk, K = dk),
// so that the epilogue thread n owns column n of S: the seam updates stay
// thread-local.  A = S^T sits in tensor memory, B = Qhat_j^T in shared memory,
// both fp16 split into hi + lo (lo scaled by 2^11, after exact power-of-two
// normalisation of each operand); three MMAs (hi*hi, hi*lo + lo*hi) with fp32
// accumulators give the product to about fp32 accuracy.
//
// Warp roles (384 threads): warp 0 MMA issuer, warp 1 producer (the seam window
// of each position -- k, q, v tiles by TMA, beta and alpha by lane loads -- into
// one of two shared-memory slots, then the Qhat_j and S_j tiles, fp32, plus an
// L2 prefetch one position further), warps 2-3 convert Qhat_j into the B
// operand, warps 4-11 own the state (two threads per column: seam, epilogue, A
// operand).
// Tensor memory: [0,128) D hi*hi, [128,256) D cross terms, [256,320) A hi,
// [320,384) A lo (fp16 pairs, element k in the low half of column k/2).
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
constexpr uint32_t OFF_SEAM0 = 196608; // seam window slots: [k | q | v] x [w][128] inputs each
constexpr uint32_t kSeamBuf = 12288;   //   (12 KB: w <= 16 tokens in bf16, w <= 8 in fp32)
constexpr uint32_t OFF_XCH = OFF_SEAM0 + 2 * kSeamBuf;   // state pair exchange (3 KB)
constexpr uint32_t SMEM_DYN = OFF_XCH + 3072 + 1024;
constexpr uint32_t T_DM = 0, T_DC = 128, T_AH = 256, T_AL = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kLoScale = 2048.f;     // 2^11
constexpr float kLoUnscale = 1.f / 2048.f;
constexpr uint32_t kDrainLimit = 1u << 20;

enum {
  C_QFULL = 0, C_QFREE, C_SFULL, C_SFREE, C_BREADY, C_AREADY, C_DDONE, C_DRAIN,
  C_WFULL0, C_WFULL1, C_WFREE0, C_WFREE1, C_COUNT
};

struct CCtl {
  uint64_t bar[C_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t qexp[2];      // power-of-two exponent of max|Qhat_j| (ring by position parity)
  uint32_t qmax;        // converter: max |Qhat| bits
  uint32_t smax;        // epilogue: max |S| bits
  float sbeta[2][16];   // seam window slots: beta_t and alpha_t = e^{g_t}
  float salpha[2][16];
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// x with the mantissa truncated to 10 stored bits (11 significant): exact in fp16
// whenever x is in fp16's normal range
__device__ __forceinline__ float trunc11(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// four consecutive inputs from a shared-memory seam slot, as fp32
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
// 32 lanes x 16 consecutive columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void tma_load_3d_c(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
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
// exponent e with 2^e <= m < 2^(e+1) (m > 0); 0 for m == 0
__device__ __forceinline__ int floor_log2(float m) {
  if (!(m > 0.f)) return 0;
  int e;
  frexpf(m, &e);
  return e - 1;
}

}  // namespace

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
    compose_tc_kernel(const __grid_constant__ ComposeParams p,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_s,
                      const __grid_constant__ CUtensorMap tm_wk,
                      const __grid_constant__ CUtensorMap tm_wq,
                      const __grid_constant__ CUtensorMap tm_wv) {
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
  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    for (int i = 0; i < C_COUNT; ++i) mbar_init(BAR(i), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_s);
    if (p.w > 0) {
      prefetch_tmap(&tm_wk);
      prefetch_tmap(&tm_wq);
      prefetch_tmap(&tm_wv);
    }
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t limit = p.spin_limit;
  auto wait_k = [&](int i, uint32_t k) -> bool {
    const uint32_t b = BAR(i), par = k & 1u;
    for (uint32_t n = 0; n < limit; ++n) {
      if (mbar_try(b, par)) return true;
      if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
    }
    if (atomicExch(&ctl.abort_flag, 1) == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, 200 + i);
    return false;
  };
  // segment of position j, or -1 when out of range (that position is skipped)
  auto seg_at = [&](int j) -> int {
    const int sg = p.order[static_cast<int64_t>(r) * P + j];
    return (sg >= 0 && sg < p.n_seg) ? sg : -1;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < P && ok; ++j) {
        if (!(ok = wait_k(C_AREADY, j) && wait_k(C_BREADY, j))) break;
        tc_fence_after();
        if (seg_at(j) >= 0) {
          const uint32_t id = idesc_f16(128, 128);
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t bo = (ks >> 2) * 16384 + (ks & 3) * 32;
            const uint64_t bh = desc_sw128(sb + OFF_BH + bo), bl = desc_sw128(sb + OFF_BL + bo);
            mma_ts(tmem + T_DM, tmem + T_AH + ks * 8, bh, id, ks > 0);
            mma_ts(tmem + T_DC, tmem + T_AH + ks * 8, bl, id, ks > 0);
            mma_ts(tmem + T_DC, tmem + T_AL + ks * 8, bh, id, 1);
          }
        }
        mma_commit(BAR(C_DDONE));
      }
      if (!ok) {
        mma_commit(BAR(C_DRAIN));
        mbar_wait(BAR(C_DRAIN), 0, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- producer
    // per position j: the seam window into slot j & 1 (once the state role has
    // released the window two positions back), then Qhat_j and S_j
    bool ok = true;
    uint32_t qiss = 0, siss = 0, wiss0 = 0, wiss1 = 0;
    const int w = p.w;
    const uint32_t wbytes = static_cast<uint32_t>(w) * kD * sizeof(Tin);
    for (int j = 0; j < P && ok; ++j) {
      const int sg = seg_at(j);
      if (w > 0) {
        const uint32_t b = j & 1;
        bool f = (lane == 0) && j >= 2 && !wait_k(C_WFREE0 + b, (j >> 1) - 1);
        if (__shfl_sync(0xffffffffu, f, 0)) { ok = false; break; }
        const int32_t tok0 = (r * P + j) * w;
        if (lane < w) {
          const int64_t tk = (static_cast<int64_t>(tok0) + lane) * S + s;
          ctl.sbeta[b][lane] = p.beta[tk];
          ctl.salpha[b][lane] = __expf(p.log_alpha[tk]);
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t dst = sb + OFF_SEAM0 + b * kSeamBuf, bar = BAR(C_WFULL0 + b);
          mbar_expect_tx(bar, 3 * wbytes);
          tma_load_3d_c(dst, &tm_wk, bar, 0, s, tok0);
          tma_load_3d_c(dst + wbytes, &tm_wq, bar, 0, s, tok0);
          tma_load_3d_c(dst + 2 * wbytes, &tm_wv, bar, 0, s, tok0);
          if (b) ++wiss1; else ++wiss0;
        }
      }
      if (lane == 0) {
        if (j + 1 < P) {  // next position's tiles towards L2
          const int sn = seg_at(j + 1);
          if (sn >= 0) {
            const int32_t row = (sn * S + s) * kD;
            l2_prefetch_2d(&tm_q, 0, row);
            l2_prefetch_2d(&tm_s, 0, row);
          }
        }
        if (j >= 1 && !wait_k(C_QFREE, j - 1)) {
          ok = false;
        } else {
          if (sg >= 0) {
            mbar_expect_tx(BAR(C_QFULL), kD * kD * 4);
            tma_load_2d(sb + OFF_QS, &tm_q, BAR(C_QFULL), 0, (sg * S + s) * kD);
          } else {
            mbar_arrive(BAR(C_QFULL));
          }
          ++qiss;
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
      if (wiss0) mbar_wait(BAR(C_WFULL0), (wiss0 - 1) & 1u, kDrainLimit);
      if (wiss1) mbar_wait(BAR(C_WFULL1), (wiss1 - 1) & 1u, kDrainLimit);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- converter
    const int ct = tid - 64;  // 0..63
    bool ok = true;
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
      // B is free once the previous position's MMAs are done
      fail = (ct == 0) && j >= 1 && !wait_k(C_DDONE, j - 1);
      if (named_or(1, 64, fail)) { ok = false; break; }
      if (sg >= 0) {
        const float sc = ldexpf(1.f, -ea);
#pragma unroll 4
        for (int e = ct; e < 4096; e += 64) {
          const int i = e >> 5, k4 = e & 31;         // row i, k = 4*k4 .. 4*k4+3
          const float4 v = reinterpret_cast<const float4*>(qs)[e];
          const float a0 = v.x * sc, a1 = v.y * sc, a2 = v.z * sc, a3 = v.w * sc;
          // hi keeps the top 11 significant bits (exact in fp16 for the
          // normalised range), lo = fp16((a - hi) 2^11) with a - hi exact in fp32
          const float t0 = trunc11(a0), t1 = trunc11(a1), t2 = trunc11(a2), t3 = trunc11(a3);
          const __half2 h01 = __floats2half2_rn(t0, t1), h23 = __floats2half2_rn(t2, t3);
          const __half2 l01 = __floats2half2_rn((a0 - t0) * kLoScale, (a1 - t1) * kLoScale);
          const __half2 l23 = __floats2half2_rn((a2 - t2) * kLoScale, (a3 - t3) * kLoScale);
          const uint32_t off = sw128_off(i, 4 * k4, 128);    // 8-byte aligned half chunk
          *reinterpret_cast<uint2*>(sm + OFF_BH + off) = make_uint2(h2u(h01), h2u(h23));
          *reinterpret_cast<uint2*>(sm + OFF_BL + off) = make_uint2(h2u(l01), h2u(l23));
        }
      }
      if (ct == 0) ctl.qexp[j & 1] = ea;
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
    // 64..127; TMEM lane = n).  The seam's per-token dot products k^T S[:,n] and
    // o_n = S[:,n]^T q are split over the pair and combined through a small
    // exchange area (double-buffered by token parity, one barrier per token).
    const int n = (warp & 3) * 32 + lane;        // column n of S = TMEM lane
    const int h = (warp - 4) >> 2;               // row half
    const int i0 = 64 * h;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int et = tid - 128;                     // 0..255
    const int64_t st_base = (static_cast<int64_t>(r) * S + s) * kD * kD;
    float* xu = reinterpret_cast<float*>(sm + OFF_XCH);   // [2 parity][2 half][128] partial k^T S
    float* xo = xu + 2 * 2 * kD;                          // [2 parity][128] partial o (row half 1)
    float x[kH];
#pragma unroll
    for (int i = 0; i < kH; ++i) x[i] = p.state_in ? p.state_in[st_base + (i0 + i) * kD + n] : 0.f;
    bool ok = true;
    for (int j = 0; j < P && ok; ++j) {
      const int sg = seg_at(j);
      if (sg < 0 && et == 0) report(p.ws, HYPIC_ERR_INDEX, 210);
      // ---- seam window of position j (fp32)
      if (p.w > 0) {
        const int64_t tok0 = (static_cast<int64_t>(r) * P + j) * p.w;
        const uint32_t b = j & 1;
        bool wf = (et == 0) && !wait_k(C_WFULL0 + b, j >> 1);
        if (named_or(2, 256, wf)) { ok = false; break; }
        const Tin* kw = reinterpret_cast<const Tin*>(sm + OFF_SEAM0 + b * kSeamBuf);
        const Tin* qw = kw + p.w * kD;
        const Tin* vw = qw + p.w * kD;
        // the token decays are applied lazily: the true column is dsc * x, with
        // dsc the product of alpha over the window so far (one multiply per
        // element at the end of the window instead of one per element per token)
        float dsc = 1.f;
        float o_prev = 0.f;   // row half 0: its partial o of the previous token
        for (int t = 0; t < p.w; ++t) {
          const int tp = t & 1;
          const float be = ctl.sbeta[b][t], al = ctl.salpha[b][t];
          const float vn = ld1(vw + t * kD + n);
          const Tin* kv = kw + t * kD + i0;
          const Tin* qv = qw + t * kD + i0;
          float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
          for (int i = 0; i < kH; i += 4) {
            const float4 k4 = ld4(kv + i);
            u0 = fmaf(k4.x, x[i], u0);
            u1 = fmaf(k4.y, x[i + 1], u1);
            u2 = fmaf(k4.z, x[i + 2], u2);
            u3 = fmaf(k4.w, x[i + 3], u3);
          }
          xu[(tp * 2 + h) * kD + n] = (u0 + u1) + (u2 + u3);
          named_sync(2, 256);
          // the partner's half of k^T S; and the previous token's o from row half 1
          const float u = xu[(tp * 2 + h) * kD + n] + xu[(tp * 2 + (h ^ 1)) * kD + n];
          if (h == 0 && t > 0) {
            const int64_t tkp = (tok0 + t - 1) * S + s;
            store_o(p, tkp * kD + n, o_prev + xo[(tp ^ 1) * kD + n]);
          }
          // true update: S <- al (S - be k (k^T S)) + be k v^T; with S = dsc x and
          // dsc' = dsc al:  x <- x + k cc / dsc',  cc = be vn - al be (k^T S)
          const float cc = be * vn - al * be * (dsc * u);
          dsc *= al;
          if (dsc < 0x1p-60f) {   // strong decay: fold the factor in before it underflows
#pragma unroll
            for (int i = 0; i < kH; ++i) x[i] *= dsc;
            dsc = 1.f;
          }
          const float ccs = cc / dsc;
          float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
          for (int i = 0; i < kH; i += 4) {
            const float4 k4 = ld4(kv + i);
            const float4 q4 = ld4(qv + i);
            x[i] = fmaf(k4.x, ccs, x[i]);
            x[i + 1] = fmaf(k4.y, ccs, x[i + 1]);
            x[i + 2] = fmaf(k4.z, ccs, x[i + 2]);
            x[i + 3] = fmaf(k4.w, ccs, x[i + 3]);
            o0 = fmaf(q4.x, x[i], o0);
            o1 = fmaf(q4.y, x[i + 1], o1);
            o2 = fmaf(q4.z, x[i + 2], o2);
            o3 = fmaf(q4.w, x[i + 3], o3);
          }
          const float op = dsc * ((o0 + o1) + (o2 + o3));
          if (h == 0) o_prev = op;
          else xo[tp * kD + n] = op;
        }
#pragma unroll
        for (int i = 0; i < kH; ++i) x[i] *= dsc;
        named_sync(2, 256);  // the slot is read and the last o half is in the exchange
        if (h == 0) {
          const int tl = p.w - 1;
          store_o(p, ((tok0 + tl) * S + s) * kD + n, o_prev + xo[(tl & 1) * kD + n]);
        }
        if (et == 0) mbar_arrive(BAR(C_WFREE0 + b));
      }
      // ---- A operand: S^T rows n, columns (k) i0..i0+63 of this half,
      //      normalised by 2^-eb, fp16 hi + lo
      int eb = 0;
      if (sg >= 0) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < kH; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (et == 0) ctl.smax = 0u;
        named_sync(2, 256);
        if (lane == 0) atomicMax(&ctl.smax, __float_as_uint(m));
        named_sync(2, 256);
        eb = floor_log2(__uint_as_float(ctl.smax));
        const float sc = ldexpf(1.f, -eb);
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a0 = x[32 * bb + 2 * e] * sc, a1 = x[32 * bb + 2 * e + 1] * sc;
            const __half2 hh = __floats2half2_rn(a0, a1);
            const float2 f = __half22float2(hh);
            hi[e] = h2u(hh);
            lo[e] = h2u(__floats2half2_rn((a0 - f.x) * kLoScale, (a1 - f.y) * kLoScale));
          }
          const uint32_t col = (i0 >> 1) + 16 * bb;
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tmem + lane_off + T_AH + col),
              "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]), "r"(hi[4]), "r"(hi[5]), "r"(hi[6]),
              "r"(hi[7]), "r"(hi[8]), "r"(hi[9]), "r"(hi[10]), "r"(hi[11]), "r"(hi[12]),
              "r"(hi[13]), "r"(hi[14]), "r"(hi[15])
              : "memory");
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tmem + lane_off + T_AL + col),
              "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]), "r"(lo[4]), "r"(lo[5]), "r"(lo[6]),
              "r"(lo[7]), "r"(lo[8]), "r"(lo[9]), "r"(lo[10]), "r"(lo[11]), "r"(lo[12]),
              "r"(lo[13]), "r"(lo[14]), "r"(lo[15])
              : "memory");
        }
        tmem_wait_st();
      }
      tc_fence_before();
      named_sync(2, 256);
      if (et == 0) mbar_arrive(BAR(C_AREADY));
      // ---- epilogue: x <- c * D + S_j (column n, this row half)
      bool fail = (et == 0) && !(wait_k(C_DDONE, j) && wait_k(C_SFULL, j));
      if (named_or(2, 256, fail)) { ok = false; break; }
      tc_fence_after();
      if (sg >= 0) {
        const int64_t u = static_cast<int64_t>(sg) * S + s;
        const int ea = ctl.qexp[j & 1];
        const float c = expf(p.log_T[u] + static_cast<float>(p.exp2[u] + ea + eb) * 0.69314718055994531f);
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
      named_sync(2, 256);
      if (et == 0) mbar_arrive(BAR(C_SFREE));
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

// 3-D map over the seam inputs [n_req * n_pos * w][n_streams][128] (bf16 or fp32);
// box = one stream's 128 channels x w tokens, landing [w][128] in a slot.
bool make_map_seam(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams, int w,
                   bool f32) {
  auto fn = encode_fn_c();
  if (!fn) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(n_streams),
                        static_cast<cuuint64_t>(n_tok)};
  cuuint64_t strides[2] = {kD * es, kD * es * static_cast<cuuint64_t>(n_streams)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), 1u, static_cast<cuuint32_t>(w)};
  cuuint32_t ones[3] = {1u, 1u, 1u};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool compose_tc_supported(const ComposeParams& p) {
  // a seam window slot holds 3 x w x 128 inputs: w <= 16 in bf16, w <= 8 in fp32
  const int max_w = (p.seam_dtype == HYPIC_F32) ? 8 : 16;
  const int64_t n_seam_tok = static_cast<int64_t>(p.n_req) * p.n_pos * p.w;
  return p.kind == HYPIC_GDN && (p.w == 0 || p.seam_kind == HYPIC_GDN) && p.dk == kD &&
         p.dv == kD && p.w <= max_w && p.n_seg > 0 &&
         n_seam_tok < (int64_t{1} << 31);
}

cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t st) {
  const int64_t n_units = static_cast<int64_t>(p.n_seg) * p.n_streams;
  CUtensorMap mq, ms;
  if (!make_map_f32(&mq, p.Qhat, n_units) || !make_map_f32(&ms, p.Sc, n_units))
    return cudaErrorInvalidValue;
  const bool f32 = (p.w > 0 && p.seam_dtype == HYPIC_F32);
  CUtensorMap mwk = mq, mwq = mq, mwv = mq;   // unused without a seam window
  if (p.w > 0) {
    const int64_t n_tok = static_cast<int64_t>(p.n_req) * p.n_pos * p.w;
    if (!make_map_seam(&mwk, p.k, n_tok, p.n_streams, p.w, f32) ||
        !make_map_seam(&mwq, p.q, n_tok, p.n_streams, p.w, f32) ||
        !make_map_seam(&mwv, p.v, n_tok, p.n_streams, p.w, f32))
      return cudaErrorInvalidValue;
  }
  auto kern = f32 ? compose_tc_kernel<float> : compose_tc_kernel<__nv_bfloat16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  kern<<<p.n_req * p.n_streams, kThreads, SMEM_DYN, st>>>(p, mq, ms, mwk, mwq, mwv);
  return cudaGetLastError();
}

}  // namespace hypic
