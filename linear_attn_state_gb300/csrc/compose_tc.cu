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
// Warp roles (256 threads): warp 0 MMA issuer, warp 1 TMA producer (Qhat_j and
// S_j tiles, fp32, plus L2 prefetch one position further), warps 2-3 convert
// Qhat_j into the B operand, warps 4-7 own the state (seam, epilogue, A operand).
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
constexpr int kThreads = 256;
constexpr uint32_t OFF_QS = 0;        // Qhat_j staging fp32 [128 i][128 k] (64 KB)
constexpr uint32_t OFF_SJ = 65536;    // S_j staging fp32 [128 i][128 n] (64 KB)
constexpr uint32_t OFF_BH = 131072;   // B hi: Qhat rows i, K-major SW128, 2 K blocks (32 KB)
constexpr uint32_t OFF_BL = 163840;   // B lo (32 KB)
constexpr uint32_t OFF_SEAM = 196608; // seam vectors: k_t, q_t fp32 [w][128] each (<= 16 KB)
constexpr int kMaxW = 16;
constexpr uint32_t SMEM_DYN = OFF_SEAM + 2 * kMaxW * kD * 4 + 1024;
constexpr uint32_t T_DM = 0, T_DC = 128, T_AH = 256, T_AL = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kLoScale = 2048.f;     // 2^11
constexpr float kLoUnscale = 1.f / 2048.f;
constexpr uint32_t kDrainLimit = 1u << 20;

enum { C_QFULL = 0, C_QFREE, C_SFULL, C_SFREE, C_BREADY, C_AREADY, C_DDONE, C_DRAIN, C_COUNT };

struct CCtl {
  uint64_t bar[C_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t qexp[2];      // power-of-two exponent of max|Qhat_j| (ring by position parity)
  uint32_t qmax;        // converter: max |Qhat| bits
  uint32_t smax;        // epilogue: max |S| bits
};

template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

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
  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    for (int i = 0; i < C_COUNT; ++i) mbar_init(BAR(i), 1);
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
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t qiss = 0, siss = 0;
      for (int j = 0; j < P && ok; ++j) {
        const int sg = seg_at(j);
        if (j + 1 < P) {  // next position's tiles towards L2
          const int sn = seg_at(j + 1);
          if (sn >= 0) {
            const int32_t row = (sn * S + s) * kD;
            l2_prefetch_2d(&tm_q, 0, row);
            l2_prefetch_2d(&tm_s, 0, row);
          }
        }
        if (j >= 1 && !(ok = wait_k(C_QFREE, j - 1))) break;
        if (sg >= 0) {
          mbar_expect_tx(BAR(C_QFULL), kD * kD * 4);
          tma_load_2d(sb + OFF_QS, &tm_q, BAR(C_QFULL), 0, (sg * S + s) * kD);
        } else {
          mbar_arrive(BAR(C_QFULL));
        }
        ++qiss;
        if (j >= 1 && !(ok = wait_k(C_SFREE, j - 1))) break;
        if (sg >= 0) {
          mbar_expect_tx(BAR(C_SFULL), kD * kD * 4);
          tma_load_2d(sb + OFF_SJ, &tm_s, BAR(C_SFULL), 0, (sg * S + s) * kD);
        } else {
          mbar_arrive(BAR(C_SFULL));
        }
        ++siss;
      }
      if (!ok) {
        if (qiss) mbar_wait(BAR(C_QFULL), (qiss - 1) & 1u, kDrainLimit);
        if (siss) mbar_wait(BAR(C_SFULL), (siss - 1) & 1u, kDrainLimit);
      }
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
          const __half2 h01 = __floats2half2_rn(a0, a1), h23 = __floats2half2_rn(a2, a3);
          const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
          const __half2 l01 = __floats2half2_rn((a0 - f01.x) * kLoScale, (a1 - f01.y) * kLoScale);
          const __half2 l23 = __floats2half2_rn((a2 - f23.x) * kLoScale, (a3 - f23.y) * kLoScale);
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
    // ---------------------------------------------------------------- state owner
    const int n = (warp & 3) * 32 + lane;      // column n of S = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int et = tid - 128;                   // 0..127
    float* seam_k = reinterpret_cast<float*>(sm + OFF_SEAM);
    float* seam_q = seam_k + kMaxW * kD;
    const Tin* qp = static_cast<const Tin*>(p.q);
    const Tin* kp = static_cast<const Tin*>(p.k);
    const Tin* vp = static_cast<const Tin*>(p.v);
    const int64_t st_base = (static_cast<int64_t>(r) * S + s) * kD * kD;
    float x[kD];
#pragma unroll
    for (int i = 0; i < kD; ++i) x[i] = p.state_in ? p.state_in[st_base + i * kD + n] : 0.f;
    bool ok = true;
    for (int j = 0; j < P && ok; ++j) {
      const int sg = seg_at(j);
      if (sg < 0 && et == 0) report(p.ws, HYPIC_ERR_INDEX, 210);
      // ---- seam window of position j (fp32, thread-local column)
      if (p.w > 0) {
        const int64_t tok0 = (static_cast<int64_t>(r) * P + j) * p.w;
        named_sync(2, 128);  // previous tokens' vectors consumed
        for (int t = 0; t < p.w; ++t) {
          const int64_t tk = (tok0 + t) * S + s;
          seam_k[t * kD + et] = ldf(kp, tk * kD + et);
          seam_q[t * kD + et] = ldf(qp, tk * kD + et);
        }
        named_sync(2, 128);
        for (int t = 0; t < p.w; ++t) {
          const int64_t tk = (tok0 + t) * S + s;
          const float be = p.beta[tk], al = __expf(p.log_alpha[tk]);
          const float vn = ldf(vp, tk * kD + n);
          const float* kv = seam_k + t * kD;
          const float* qv = seam_q + t * kD;
          float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
          for (int i = 0; i < kD; i += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kv + i);
            u0 = fmaf(k4.x, x[i], u0);
            u1 = fmaf(k4.y, x[i + 1], u1);
            u2 = fmaf(k4.z, x[i + 2], u2);
            u3 = fmaf(k4.w, x[i + 3], u3);
          }
          const float cc = be * vn - al * be * ((u0 + u1) + (u2 + u3));
          float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
          for (int i = 0; i < kD; i += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kv + i);
            const float4 q4 = *reinterpret_cast<const float4*>(qv + i);
            x[i] = fmaf(al, x[i], k4.x * cc);
            x[i + 1] = fmaf(al, x[i + 1], k4.y * cc);
            x[i + 2] = fmaf(al, x[i + 2], k4.z * cc);
            x[i + 3] = fmaf(al, x[i + 3], k4.w * cc);
            o0 = fmaf(q4.x, x[i], o0);
            o1 = fmaf(q4.y, x[i + 1], o1);
            o2 = fmaf(q4.z, x[i + 2], o2);
            o3 = fmaf(q4.w, x[i + 3], o3);
          }
          p.out_o[tk * kD + n] = (o0 + o1) + (o2 + o3);
        }
      }
      // ---- A operand: S^T row n (this column), normalised by 2^-eb, fp16 hi + lo
      int eb = 0;
      if (sg >= 0) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < kD; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (et == 0) ctl.smax = 0u;
        named_sync(2, 128);
        if (lane == 0) atomicMax(&ctl.smax, __float_as_uint(m));
        named_sync(2, 128);
        eb = floor_log2(__uint_as_float(ctl.smax));
        const float sc = ldexpf(1.f, -eb);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a0 = x[32 * b + 2 * e] * sc, a1 = x[32 * b + 2 * e + 1] * sc;
            const __half2 h = __floats2half2_rn(a0, a1);
            const float2 f = __half22float2(h);
            hi[e] = h2u(h);
            lo[e] = h2u(__floats2half2_rn((a0 - f.x) * kLoScale, (a1 - f.y) * kLoScale));
          }
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tmem + lane_off + T_AH + 16 * b),
              "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3]), "r"(hi[4]), "r"(hi[5]), "r"(hi[6]),
              "r"(hi[7]), "r"(hi[8]), "r"(hi[9]), "r"(hi[10]), "r"(hi[11]), "r"(hi[12]),
              "r"(hi[13]), "r"(hi[14]), "r"(hi[15])
              : "memory");
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tmem + lane_off + T_AL + 16 * b),
              "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]), "r"(lo[4]), "r"(lo[5]), "r"(lo[6]),
              "r"(lo[7]), "r"(lo[8]), "r"(lo[9]), "r"(lo[10]), "r"(lo[11]), "r"(lo[12]),
              "r"(lo[13]), "r"(lo[14]), "r"(lo[15])
              : "memory");
        }
        tmem_wait_st();
      }
      tc_fence_before();
      named_sync(2, 128);
      if (et == 0) mbar_arrive(BAR(C_AREADY));
      // ---- epilogue: x <- c * D + S_j (column n)
      bool fail = (et == 0) && !(wait_k(C_DDONE, j) && wait_k(C_SFULL, j));
      if (named_or(2, 128, fail)) { ok = false; break; }
      tc_fence_after();
      if (sg >= 0) {
        const int64_t u = static_cast<int64_t>(sg) * S + s;
        const int ea = ctl.qexp[j & 1];
        const float c = expf(p.log_T[u] + static_cast<float>(p.exp2[u] + ea + eb) * 0.69314718055994531f);
        const float* sj = reinterpret_cast<const float*>(sm + OFF_SJ);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t dm[32], dc[32];
          tmem_ld32(tmem + lane_off + T_DM + 32 * b, dm);
          tmem_ld32(tmem + lane_off + T_DC + 32 * b, dc);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int i = 32 * b + e;
            const float d = __uint_as_float(dm[e]) + __uint_as_float(dc[e]) * kLoUnscale;
            x[i] = fmaf(c, d, sj[i * kD + n]);
          }
        }
      }
      tc_fence_before();
      named_sync(2, 128);
      if (et == 0) mbar_arrive(BAR(C_SFREE));
    }
    if (ok) {
      float* out = p.state_out + st_base;
#pragma unroll
      for (int i = 0; i < kD; ++i) out[i * kD + n] = x[i];
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
  return p.kind == HYPIC_GDN && p.dk == kD && p.dv == kD && p.w <= kMaxW && p.n_seg > 0;
}

cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t st) {
  const int64_t n_units = static_cast<int64_t>(p.n_seg) * p.n_streams;
  CUtensorMap mq, ms;
  if (!make_map_f32(&mq, p.Qhat, n_units) || !make_map_f32(&ms, p.Sc, n_units))
    return cudaErrorInvalidValue;
  const bool f32 = (p.w > 0 && p.seam_dtype == HYPIC_F32);
  auto kern = f32 ? compose_tc_kernel<float> : compose_tc_kernel<__nv_bfloat16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  kern<<<p.n_req * p.n_streams, kThreads, SMEM_DYN, st>>>(p, mq, ms);
  return cudaGetLastError();
}

}  // namespace hypic
