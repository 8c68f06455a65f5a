// Chunked gated-delta segment build on tcgen05 tensor cores (sm_103a).
//
// What it computes (youleyou.com HYPIC article, linear-layer paragraph): for
// every (segment, stream) unit the pair T_C = A_L ... A_1 and S(C|0), with
// A_t = alpha_t (I - beta_t k_t k_t^T) and S_t = A_t S_{t-1} + beta_t k_t v_t^T.
// T is carried factored, T = exp(log_T) 2^exp2 Qhat, Q = H_L ... H_1 with
// H_t = I - beta_t k_t k_t^T (decay summed in log space, Q rescaled by exact
// powers of two), so long segments stay in fp32 range.
//
// Chunked WY/UT form (64 tokens per chunk, c_i = within-chunk cumulative
// log-decay, Gamma_i = e^{c_i}):
//   G   = K K^T
//   L_Q = strictly-lower(diag(beta) G),  L_S = strictly-lower(diag(beta) G e^{c_i - c_j})
//   W   = (I + L_Q)^-1 diag(beta) K,    U = (I + L_S)^-1 diag(beta) V
//   X   = [Q | S] (dk x (dk+dv));  S is pre-scaled by the chunk's Gamma_n:
//   P   = W Xhat,  R = [ -P_Q | diag(Gamma_n / Gamma_i) U - P_S ],  X += K^T R
// Every contraction is a tcgen05.mma (kind::f16, fp16 operands from shared
// memory, fp32 accumulators in tensor memory); the two 64x64 unit-triangular
// inverses are fp32 column solves on CUDA cores.  K and V tiles arrive by TMA
// (one chunk ahead).  The state X stays in tensor memory for the whole unit.
//
// One CTA per SM, persistent, 128 threads (thread i <-> tensor-memory lane i);
// work items are popped in longest-body-first order from the device queue.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,256) X   [256,320) G then P_Q^T   [320,384) P_S^T   [384,448) W^T   [448,512) U^T
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "hypic_internal.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kC = 64;        // chunk length
constexpr int kD = 128;       // dk = dv
constexpr int kThreads = 128;

// Dynamic shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_STG_K = 0;        // TMA staging, bf16 [64 t][128 d]
constexpr uint32_t OFF_STG_V = 16384;
constexpr uint32_t OFF_KT = 32768;       // K   [t][d]  K-major SW128, 64 rows, 2 K blocks
constexpr uint32_t OFF_KTT = 49152;      // K^T [d][t]  128 rows, 1 K block
constexpr uint32_t OFF_VT = 65536;       // V^T [d][t]  128 rows, 1 K block
constexpr uint32_t OFF_BW = 81920;       // beta_j Inv_Q[t][j] as [t][j], 64 rows
constexpr uint32_t OFF_BU = 90112;       // beta_j Inv_S[t][j] as [t][j], 64 rows
constexpr uint32_t OFF_WT = 98304;       // W [t][d], 64 rows, 2 K blocks
constexpr uint32_t OFF_XH = 114688;      // Xhat^T [n][i], 256 rows, 2 K blocks
constexpr uint32_t OFF_RB = 180224;      // R^T [n][t], 256 rows, 1 K block (32 KB)
constexpr uint32_t LROW = 68;            // fp32 row stride of L_Q / L_S during the solve
constexpr uint32_t OFF_LQ = OFF_RB;                       // L_Q fp32 [64][68] (aliases R)
constexpr uint32_t OFF_LS = OFF_RB + 64 * LROW * 4;       // L_S fp32 [64][68]
constexpr uint32_t SMEM_END = OFF_LS + 64 * LROW * 4;     // 215040
constexpr uint32_t SMEM_DYN = SMEM_END + 1024;            // + alignment slack

constexpr uint32_t T_X = 0, T_G = 256, T_PQ = 256, T_PS = 320, T_W = 384, T_U = 448;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDrainLimit = 1u << 26;

__device__ __forceinline__ uint16_t h16(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  return static_cast<uint32_t>(h16(a)) | (static_cast<uint32_t>(h16(b)) << 16);
}

__device__ __forceinline__ void st_u16(uint8_t* sm, uint32_t off, uint16_t v) {
  *reinterpret_cast<uint16_t*>(sm + off) = v;
}

// bf16 pair (packed in 32 bits) -> fp16 pair
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w, bool keep) {
  if (!keep) return 0u;
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_h2(lo, hi);
}

struct Ctl {
  uint64_t bar_tma;
  uint64_t bar_mma;
  uint32_t tmem_base;
  int32_t item;
  float cs[kC];       // within-chunk cumulative log-decay
  float beta[kC];
  float gsum_next;    // log-decay sum of the next chunk
  float wsum[2];      // warp totals of the within-chunk scan
  float nsum[2];      // warp partial sums of the next chunk's log-decay
  uint32_t qmax[2];   // max |Qhat| bits, alternating between passes
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    gdn_build_tc_kernel(const __grid_constant__ BuildParams p,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ Ctl ctl;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const int S = p.n_streams;

  if (p.ws->status != 0) return;  // the work list is not valid

  const uint32_t bar_tma = smem_u32(&ctl.bar_tma);
  const uint32_t bar_mma = smem_u32(&ctl.bar_mma);
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  uint32_t ph_tma = 0, ph_mma = 0;
  bool tma_pending = false, mma_pending = false, aborted = false;
  const uint32_t limit = p.spin_limit;

  // Waits on an mbarrier phase with a bounded poll; the decision is made
  // block-uniform so that every thread takes the same path.
  auto wait_bar = [&](uint32_t bar, uint32_t& ph, bool& pending, int site) -> bool {
    const bool ok = mbar_wait(bar, ph, limit);
    const bool any_fail = __syncthreads_or(!ok);
    if (any_fail) {
      if (tid == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, site);
      aborted = true;
      return false;
    }
    ph ^= 1u;
    pending = false;
    return true;
  };

  for (;;) {
    if (tid == 0) ctl.item = static_cast<int32_t>(atomicAdd(&p.ws->queue, 1u));
    __syncthreads();
    const int idx = ctl.item;
    __syncthreads();
    if (idx >= p.n_items) break;
    const WorkItem it = p.items[idx];
    const int64_t u = it.unit;
    const int s = it.unit % S;
    float* __restrict__ Qg = p.Qhat + u * kD * kD;
    float* __restrict__ Sg = p.S + u * kD * kD;

    if (it.len == 0) {  // identity pair
      for (int e = tid; e < kD * kD; e += kThreads) {
        Qg[e] = ((e / kD) == (e % kD)) ? 1.f : 0.f;
        Sg[e] = 0.f;
      }
      if (tid == 0) {
        p.exp2[u] = 0;
        p.log_T[u] = 0.f;
      }
      continue;
    }
    const int nc = (it.len + kC - 1) / kC;

    // ---- initial state: X = [I | 0] in tensor memory, Xhat in shared memory
    {
      uint32_t r[32];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = (b * 32 + e == tid) ? 0x3f800000u : 0u;
        tmem_st32(tmem + lane_off + T_X + 32 * b, r);
      }
      tmem_wait_st();
      uint4* xh = reinterpret_cast<uint4*>(sm + OFF_XH);
      for (int e = tid; e < 65536 / 16; e += kThreads) xh[e] = make_uint4(0, 0, 0, 0);
      if (tid == 0) {
        ctl.qmax[0] = __float_as_uint(1.f);
        ctl.qmax[1] = 0u;
      }
      __syncthreads();
      st_u16(sm, OFF_XH + sw128_off(tid, tid, 256), 0x3C00u);  // 1.0 on the Q diagonal
    }
    if (tid == 0) {
      mbar_expect_tx(bar_tma, 2u * kC * kD * 2u);
      tma_load_3d(sb + OFF_STG_K, &tm_k, bar_tma, 0, s, static_cast<int32_t>(it.tok_start));
      tma_load_3d(sb + OFF_STG_V, &tm_v, bar_tma, 0, s, static_cast<int32_t>(it.tok_start));
    }
    tma_pending = true;

    double logG = 0.0;
    int exp2_acc = 0;

    for (int c = 0; c < nc && !aborted; ++c) {
      const int64_t t0 = it.tok_start + static_cast<int64_t>(c) * kC;
      const int n = min(kC, it.len - c * kC);
      const int n_next = (c + 1 < nc) ? min(kC, it.len - (c + 1) * kC) : 0;

      // (a) beta, within-chunk cumulative log-decay; next chunk's decay sum
      if (tid < kC) {
        const bool v = tid < n;
        const float b = v ? p.beta[(t0 + tid) * S + s] : 0.f;
        float g = v ? p.log_alpha[(t0 + tid) * S + s] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, g, o);
          if ((tid & 31) >= o) g += y;
        }
        ctl.beta[tid] = b;
        ctl.cs[tid] = g;
        if ((tid & 31) == 31) ctl.wsum[tid >> 5] = g;
      } else {
        const int tt = tid - kC;
        float g = (tt < n_next) ? p.log_alpha[(t0 + kC + tt) * S + s] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
        if ((tid & 31) == 0) ctl.nsum[(tid - kC) >> 5] = g;
      }
      __syncthreads();
      if (tid >= 32 && tid < kC) ctl.cs[tid] += ctl.wsum[0];
      if (tid == 0) {
        ctl.qmax[(c + 1) & 1] = 0u;
        ctl.gsum_next = ctl.nsum[0] + ctl.nsum[1];
      }

      // (b) K, V of this chunk
      if (!wait_bar(bar_tma, ph_tma, tma_pending, 1)) break;

      // (c) bf16 -> fp16 in the operand layouts; rows t >= n are zero
      //     (identity tokens: k = v = 0, beta = 0, g = 0 leave the pair unchanged)
      for (int j = tid; j < kC * 16; j += kThreads) {
        const int t = j >> 4, c8 = j & 15;
        const bool keep = t < n;
        const uint4 kw = *reinterpret_cast<const uint4*>(sm + OFF_STG_K + t * 256 + c8 * 16);
        const uint4 vw = *reinterpret_cast<const uint4*>(sm + OFF_STG_V + t * 256 + c8 * 16);
        uint4 kh, vh;
        kh.x = bf2_to_h2(kw.x, keep); kh.y = bf2_to_h2(kw.y, keep);
        kh.z = bf2_to_h2(kw.z, keep); kh.w = bf2_to_h2(kw.w, keep);
        vh.x = bf2_to_h2(vw.x, keep); vh.y = bf2_to_h2(vw.y, keep);
        vh.z = bf2_to_h2(vw.z, keep); vh.w = bf2_to_h2(vw.w, keep);
        *reinterpret_cast<uint4*>(sm + OFF_KT + sw128_chunk(t, c8, 64)) = kh;
        const uint32_t kk[4] = {kh.x, kh.y, kh.z, kh.w};
        const uint32_t vv[4] = {vh.x, vh.y, vh.z, vh.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = c8 * 8 + 2 * e;
          st_u16(sm, OFF_KTT + sw128_off(d, t, 128), static_cast<uint16_t>(kk[e] & 0xFFFFu));
          st_u16(sm, OFF_KTT + sw128_off(d + 1, t, 128), static_cast<uint16_t>(kk[e] >> 16));
          st_u16(sm, OFF_VT + sw128_off(d, t, 128), static_cast<uint16_t>(vv[e] & 0xFFFFu));
          st_u16(sm, OFF_VT + sw128_off(d + 1, t, 128), static_cast<uint16_t>(vv[e] >> 16));
        }
      }
      fence_proxy_async();
      __syncthreads();

      // (d) prefetch the next chunk into the staging buffers (free now)
      if (c + 1 < nc) {
        if (tid == 0) {
          mbar_expect_tx(bar_tma, 2u * kC * kD * 2u);
          tma_load_3d(sb + OFF_STG_K, &tm_k, bar_tma, 0, s, static_cast<int32_t>(t0 + kC));
          tma_load_3d(sb + OFF_STG_V, &tm_v, bar_tma, 0, s, static_cast<int32_t>(t0 + kC));
        }
        tma_pending = true;
      }

      // (e) G = K K^T (M = 128: rows 64..127 are ignored)
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_f16(128, 64);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = OFF_KT + (ks >> 2) * 8192 + (ks & 3) * 32;
          mma_f16(tmem + T_G, desc_sw128(sb + off), desc_sw128(sb + off), id, ks > 0);
        }
        mma_commit(bar_mma);
      }
      mma_pending = true;
      if (!wait_bar(bar_mma, ph_mma, mma_pending, 2)) break;
      tc_fence_after();

      // (f) L_Q, L_S rows (thread t = token row of G)
      if (warp < 2) {
        uint32_t g0[32], g1[32];
        tmem_ld32(tmem + lane_off + T_G, g0);
        tmem_ld32(tmem + lane_off + T_G + 32, g1);
        tmem_wait_ld();
        const int t = tid;
        const float bt = ctl.beta[t], ct = ctl.cs[t];
        float* LQ = reinterpret_cast<float*>(sm + OFF_LQ) + t * LROW;
        float* LS = reinterpret_cast<float*>(sm + OFF_LS) + t * LROW;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float gv = __uint_as_float(j < 32 ? g0[j] : g1[j - 32]);
          const float lq = (j < t) ? bt * gv : 0.f;
          LQ[j] = lq;
          LS[j] = (j < t) ? lq * __expf(ct - ctl.cs[j]) : 0.f;
        }
      }
      __syncthreads();

      // (g) unit lower-triangular inverses, one column per thread:
      //     warps 0-1: (I + L_Q)^-1, warps 2-3: (I + L_S)^-1
      {
        const int j = tid & 63;
        const float* L = reinterpret_cast<const float*>(sm + (tid < 64 ? OFF_LQ : OFF_LS));
        float x[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float a0 = (i == j) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int m = 0; m + 3 < i; m += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + i * LROW + m);
            a0 = fmaf(-l4.x, x[m], a0);
            a1 = fmaf(-l4.y, x[m + 1], a1);
            a2 = fmaf(-l4.z, x[m + 2], a2);
            a3 = fmaf(-l4.w, x[m + 3], a3);
          }
#pragma unroll
          for (int m = (i & ~3); m < i; ++m) a0 = fmaf(-L[i * LROW + m], x[m], a0);
          x[i] = (i < j) ? 0.f : ((a0 + a1) + (a2 + a3));
        }
        const float bj = ctl.beta[j];
        const uint32_t dst = (tid < 64) ? OFF_BW : OFF_BU;
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 64; ++t) st_u16(sm, dst + sw128_off(t, j, 64), h16(bj * x[t]));
      }
      fence_proxy_async();
      __syncthreads();

      // (h) W^T = K^T B_W, U^T = V^T B_U (M = 128, N = 64, K = 64)
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_f16(128, 64);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_f16(tmem + T_W, desc_sw128(sb + OFF_KTT + ks * 32), desc_sw128(sb + OFF_BW + ks * 32),
                  id, ks > 0);
          mma_f16(tmem + T_U, desc_sw128(sb + OFF_VT + ks * 32), desc_sw128(sb + OFF_BU + ks * 32),
                  id, ks > 0);
        }
        mma_commit(bar_mma);
      }
      mma_pending = true;
      if (!wait_bar(bar_mma, ph_mma, mma_pending, 3)) break;
      tc_fence_after();

      // (i) W^T (lane d, column t) -> W [t][d] fp16
      {
        uint32_t w0[32], w1[32];
        tmem_ld32(tmem + lane_off + T_W, w0);
        tmem_ld32(tmem + lane_off + T_W + 32, w1);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 64; ++t)
          st_u16(sm, OFF_WT + sw128_off(t, tid, 64),
                 h16(__uint_as_float(t < 32 ? w0[t] : w1[t - 32])));
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // (j) P^T = Xhat^T W^T for the Q half and the S half (M = 128, N = 64, K = 128)
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_f16(128, 64);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
          const uint64_t bdesc = desc_sw128(sb + OFF_WT + kb * 8192 + ko);
          mma_f16(tmem + T_PQ, desc_sw128(sb + OFF_XH + kb * 32768 + ko), bdesc, id, ks > 0);
          mma_f16(tmem + T_PS, desc_sw128(sb + OFF_XH + kb * 32768 + 16384 + ko), bdesc, id,
                  ks > 0);
        }
        mma_commit(bar_mma);
      }
      mma_pending = true;
      if (!wait_bar(bar_mma, ph_mma, mma_pending, 4)) break;
      tc_fence_after();

      // (k) R^T rows: Q half -P_Q^T, S half (Gamma_n / Gamma_t) U^T - P_S^T
      {
        const float c_last = ctl.cs[kC - 1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pq[32], ps[32], uu[32];
          tmem_ld32(tmem + lane_off + T_PQ + 32 * h, pq);
          tmem_ld32(tmem + lane_off + T_PS + 32 * h, ps);
          tmem_ld32(tmem + lane_off + T_U + 32 * h, uu);
          tmem_wait_ld();
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint4 rq, rs;
            uint32_t* rqw = reinterpret_cast<uint32_t*>(&rq);
            uint32_t* rsw = reinterpret_cast<uint32_t*>(&rs);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tl = q8 * 8 + 2 * e;  // token within this half
              const int t = 32 * h + tl;
              const float f0 = __expf(c_last - ctl.cs[t]);
              const float f1 = __expf(c_last - ctl.cs[t + 1]);
              rqw[e] = pack_h2(-__uint_as_float(pq[tl]), -__uint_as_float(pq[tl + 1]));
              rsw[e] = pack_h2(f0 * __uint_as_float(uu[tl]) - __uint_as_float(ps[tl]),
                               f1 * __uint_as_float(uu[tl + 1]) - __uint_as_float(ps[tl + 1]));
            }
            const uint32_t c8 = 4 * h + q8;
            *reinterpret_cast<uint4*>(sm + OFF_RB + sw128_chunk(tid, c8, 256)) = rq;
            *reinterpret_cast<uint4*>(sm + OFF_RB + sw128_chunk(128 + tid, c8, 256)) = rs;
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // (l) X += K^T R (M = 128, N = 256, K = 64)
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_f16(128, 256);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_f16(tmem + T_X, desc_sw128(sb + OFF_KTT + ks * 32), desc_sw128(sb + OFF_RB + ks * 32),
                  id, 1u);
        mma_commit(bar_mma);
      }
      mma_pending = true;
      if (!wait_bar(bar_mma, ph_mma, mma_pending, 5)) break;
      tc_fence_after();
      if (tid == 0) logG += static_cast<double>(ctl.cs[kC - 1]);

      // (m) state pass
      if (c + 1 < nc) {
        // Q half: exact power-of-two rescale from the previous pass's max;
        // S half: pre-scaled by the next chunk's decay Gamma_n.
        int e2;
        frexpf(__uint_as_float(ctl.qmax[c & 1]), &e2);
        const int sh = 1 - e2;
        exp2_acc -= sh;
        const float sq = ldexpf(1.f, sh);
        const float gs = __expf(ctl.gsum_next);
        float mloc = 0.f;
#pragma unroll 1
        for (int b = 0; b < 8; ++b) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + T_X + 32 * b, r);
          tmem_wait_ld();
          const float sc = (b < 4) ? sq : gs;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float vv = __uint_as_float(r[e]) * sc;
            if (b < 4) mloc = fmaxf(mloc, fabsf(vv));
            r[e] = __float_as_uint(vv);
            st_u16(sm, OFF_XH + sw128_off(32 * b + e, tid, 256), h16(vv));
          }
          tmem_st32(tmem + lane_off + T_X + 32 * b, r);
        }
        tmem_wait_st();
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
        if ((tid & 31) == 0) atomicMax(&ctl.qmax[(c + 1) & 1], __float_as_uint(mloc));
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
      } else {
        // outputs: row i of Qhat and of S
#pragma unroll 1
        for (int b = 0; b < 8; ++b) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + T_X + 32 * b, r);
          tmem_wait_ld();
          float* dst = (b < 4) ? (Qg + tid * kD + 32 * b) : (Sg + tid * kD + 32 * (b - 4));
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        }
        tc_fence_before();
        __syncthreads();
      }
    }
    if (aborted) break;
    if (tid == 0) {
      p.exp2[u] = exp2_acc;
      p.log_T[u] = static_cast<float>(logG);
    }
  }

  // Teardown: on an abort, let copies and MMAs in flight land before the
  // tensor memory is released.
  if (aborted) {
    if (tma_pending) mbar_wait(bar_tma, ph_tma, kDrainLimit);
    if (mma_pending) mbar_wait(bar_mma, ph_mma, kDrainLimit);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 3-D map over [n_tok][n_streams][d] bf16; box = 64 tokens x 1 stream x d.
bool make_map(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_streams),
                        static_cast<cuuint64_t>(n_tok)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(n_streams)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1u, static_cast<cuuint32_t>(kC)};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_build_gdn_tc(const BuildParams& p, int n_sms, cudaStream_t st) {
  if (p.dk != kD || p.dv != kD) return launch_build_recurrence(p, HYPIC_BF16, st);
  CUtensorMap mk, mv;
  if (!make_map(&mk, p.k, p.n_tok, p.n_streams, kD) ||
      !make_map(&mv, p.v, p.n_tok, p.n_streams, kD))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gdn_build_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sms ? p.n_items : n_sms;
  gdn_build_tc_kernel<<<grid, kThreads, SMEM_DYN, st>>>(p, mk, mv);
  return cudaGetLastError();
}

cudaError_t launch_build_decay(const BuildParams& p, cudaStream_t st) {
  return launch_build_recurrence(p, HYPIC_BF16, st);
}

}  // namespace hypic
