// Chunked KDA segment build on tcgen05 tensor cores (sm_103a).
//
// What it computes (youleyou.com HYPIC article, linear-layer paragraph: KDA is
// one of the linear-attention families whose segment transition is cached):
// for every (segment, stream) unit the pair T_C = A_L ... A_1 and S(C|0) of the
// KDA recurrence (Kimi Linear paper, KDA section: the per-channel gate first,
// then the delta rule)
//   A_t = (I - beta_t k_t k_t^T) diag(e^{g_t}),   S_t = A_t S_{t-1} + beta_t k_t v_t^T.
//
// The gate of token t splits into its largest channel m_t and the rest
// g_t - m_t <= 0.  The cache keeps T = e^{log_T} 2^exp2 Qhat with log_T = sum m_t
// and Q = prod (I - beta k k^T) diag(e^{g - m}) (powers of two renormalise Qhat).
// Per chunk of 64 tokens, with c'_t = sum_{u<=t} (g_u - m_u) per key channel
// (all <= 0), M_t = sum_{u<=t} m_u and f_j = e^{M_n - M_j}:
//   G'  = (e^{c'} o K)(e^{-c'} o K)^T      (entry [t][s] = sum_i k_t[i] k_s[i] e^{c'_t[i] - c'_s[i]})
//   L   = strictly-lower(diag(beta) G'),   Inv = (I + L)^-1
//   W   = Inv diag(beta) (e^{c'} o K),      Kn = e^{c'_n - c'} o K
//   Q  <- diag(e^{c'_n}) Q + Kn^T R_Q,      R_Q = -W Qhat
//   S  <- e^{M_n} diag(e^{c'_n}) S + Kn^T R_S,   R_S = Inv diag(beta f) V - W (e^{M_n} S)
// The chunk start is the one reference of every decay factor: each term of G'
// is a product of two factors whose own product is at most |k_t[i] k_s[i]|, so
// rounding stays relative to the terms, while e^{-c'} alone grows with the
// chunk's decay span.  A unit with a chunk whose span exceeds kSpanLimit gets
// the exponent kKdaRedo and is rebuilt by the token recurrence right after this
// kernel (same stream); its values here are finite and discarded.
//
// The state in tensor memory is pre-scaled per channel by the next chunk's
// e^{c'_n} (and e^{M_n} for S) while the state operand of W X carries only the
// scalar part, so both the product W X and the update see the state they need.
// The contractions run on tcgen05 (kind::f16, fp32 accumulators in tensor
// memory); the key images, the B operands and R are split into bf16 hi + lo
// (three products per contraction, lo x lo dropped); the state operand and W^T
// are fp16; the 64x64 unit-triangular inverse is an fp32 blocked solve on CUDA
// cores, as in the gated-delta build.
//
// Warp roles (576 threads, one CTA per SM, persistent; the CTA takes the next
// item of the longest-first work list from a global queue when it needs one):
//   warp 0      MMA issuer (one thread) and tensor-memory owner
//   warp 1      TMA producer (one thread): the gate tile and V of each chunk;
//               takes the work items
//   warps 2-9   prep: the chunk's gates (largest gate, scans, c'), the key
//               images and Kn, L, the inverse, the B operands
//   warps 10-13 Q-chain epilogue: W^T (first half of the tokens), R_Q, the Q pass
//   warps 14-17 S-chain epilogue: W^T (second half), R_S, the S pass
// The prep of chunk g+1 (gates, key images, G', the inverse, the B operands)
// overlaps the state chain of chunk g (P, R, the updates, the passes).
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) X_Q^T  [128,256) X_S^T  [256,320) P_Q^T then R_Q^T hi/lo
//   [320,384) P_S^T (W Shat minus the decayed U term) then R_S^T hi/lo
//   [384,448) G' (lanes 64..127) then W^T
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hypic_internal.h"
#include "tc_ptx.cuh"
#include "chunk_tc.cuh"

namespace hypic {
namespace {

using namespace tc;
using namespace chunk;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 576;
constexpr float kSpanLimit = 64.f;   // largest per-channel decay span (nats) of a chunk

// ---- shared memory map (offsets from the dynamic shared memory base, which the
// kernel checks is 1024-aligned; the control block sits after the tiles) ----
constexpr uint32_t OFF_V = 0;          // V: [2 halves][64 t][64 d] bf16 SW128 (16 KB); its second
                                       // half is also the ignored rows of the G' product
constexpr uint32_t OFF_KP = 16384;     // e^{c'} o K hi, lo (16 KB each, K-tile layout)
constexpr uint32_t OFF_KPL = OFF_KP + 16384;
constexpr uint32_t OFF_KN = 49152;     // Kn = e^{c'_n - c'} o K hi, lo
constexpr uint32_t OFF_KNL = OFF_KN + 16384;
constexpr uint32_t OFF_KM = 81920;     // e^{-c'} o K hi, lo; then L / Inv, then B_W hi, lo; the
                                       // gate scan's scratch while none of them is live
constexpr uint32_t OFF_KML = OFF_KM + 16384;
constexpr uint32_t OFF_LIB = OFF_KM;                    // L / Inv fp32 [64][68]
constexpr uint32_t OFF_YT = OFF_LIB + 64 * 68 * 4;      // inverse scratch fp32 [32][36]
constexpr uint32_t OFF_BWH = OFF_KM, OFF_BWL = OFF_KM + 8192;
constexpr uint32_t OFF_MT = OFF_KM + 24576;             // largest gate per token fp32 [64]
constexpr uint32_t OFF_XQ = 114688;    // Qhat^T operand fp16, K-major [2 K blocks][128 n][64 i]
constexpr uint32_t OFF_XS = 147456;    // Shat^T operand
constexpr uint32_t OFF_WT = 180224;    // the inverse's product scratch, then -(beta f Inv)^T hi, lo
                                       // (decayed U term), then W^T fp16 MN-major [128 d][64 t]
constexpr uint32_t OFF_CP = 196608;    // the chunk's gates fp32 [4 quarters][64 t][32 i] by TMA
                                       // (128-byte swizzle), then c' in their place (32 KB)
constexpr uint32_t OFF_CTL = OFF_CP + 32768;
static_assert(OFF_YT + 32 * 36 * 4 <= OFF_MT, "inverse scratch reaches the gate-scan scratch");
static_assert(OFF_MT + 256 <= OFF_KM + 32768, "gate-scan scratch overflows its region");
constexpr uint32_t LROW = 68;

constexpr uint32_t T_XQ = 0, T_XS = 128, T_PQ = 256, T_PS = 320, T_GW = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRing = 8;
constexpr uint32_t kRingReaders = 4;        // MMA, prep, Q epilogue, S epilogue
constexpr uint32_t kDrainLimit = 1u << 20;

enum {
  B_VFULL = 0, B_VEMPTY, B_GFULL, B_CPFREE, B_IMGREADY, B_GDONE, B_BREADY, B_WDONE, B_WTREADY, B_KNREADY, B_CREADY0,
  B_CREADY1, B_XQREADY, B_XSREADY, B_PQDONE, B_PSDONE, B_RQREADY, B_RSREADY, B_UQDONE, B_USDONE,
  B_KNFREE, B_DRAIN, B_ITEMFULL0, B_ITEMEMPTY0 = B_ITEMFULL0 + kRing, B_COUNT = B_ITEMEMPTY0 + kRing
};

// Per-chunk scalars live in two slots by chunk parity: slot g & 1 is written by
// the prep for chunk g and read by the prep (beta, f) and by the epilogues
// (e^{c'_n}, M_n, the span flag) up to the pass that precedes chunk g.
struct Ctl {
  uint64_t bar[B_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
  float beta[2][kC];
  float ft[2][kC];        // f_t = e^{M_n - M_t}
  alignas(16) float gn[2][kD];   // e^{c'_n[i]} (read as float4)
  float Mn[2];            // M_n: the chunk's sum of largest gates
  int32_t bad[2];         // the chunk's decay span exceeds kSpanLimit
  uint32_t qmax[2];
  int32_t ring[kRing];
};
constexpr uint32_t SMEM_DYN = OFF_CTL + sizeof(Ctl);
static_assert(SMEM_DYN <= 232448, "shared memory over the per-block limit");

// Element (t, i) of the gate / c' tile: four 32-channel quarters of [64 t][32 i]
// (128-byte rows), the 16-byte chunks of row t permuted by XOR with t mod 8.
__device__ __forceinline__ int cpi(int t, int i) {
  return (i >> 5) * 2048 + t * 32 + ((((i & 31) >> 2) ^ (t & 7)) << 2) + (i & 3);
}

// Four 16-byte image chunks a prep thread owns: item e = pt + 256 r is token
// e >> 4 and channels 8 (e & 15) .. + 7.
__device__ __forceinline__ void load_keys(const __nv_bfloat16* __restrict__ kp, int64_t t0, int n,
                                          int S, int s, int pt, uint4 (&kv)[4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int e = pt + 256 * r, t = e >> 4, c8 = e & 15;
    kv[r] = make_uint4(0, 0, 0, 0);
    if (t < n) kv[r] = *reinterpret_cast<const uint4*>(kp + ((t0 + t) * S + s) * kD + 8 * c8);
  }
}

// bf16 pair of a 32-bit word -> floats (element a in the low half)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Key images, hi and lo, in the K-tile layout (K-major SW128, [2 d halves]
// [64 t][64 d]): element (t, i) = k[t][i] e^{x}.  MODE 0 writes both
// x = -min(c'_t[i], span bound) (at off0) and x = c'_t[i] (at off1); MODE 2
// writes x = c'_63[i] - c'_t[i] (at off0).
template <int MODE>
__device__ __forceinline__ void key_images(uint8_t* sm, uint32_t off0, uint32_t off1,
                                           const float* cp, const uint4 (&kv)[4], int pt) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int e = pt + 256 * r, t = e >> 4, c8 = e & 15;
    const float4 a0 = *reinterpret_cast<const float4*>(cp + cpi(t, 8 * c8));
    const float4 a1 = *reinterpret_cast<const float4*>(cp + cpi(t, 8 * c8 + 4));
    float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    if (MODE == 2) {
      const float4 b0 = *reinterpret_cast<const float4*>(cp + cpi(kC - 1, 8 * c8));
      const float4 b1 = *reinterpret_cast<const float4*>(cp + cpi(kC - 1, 8 * c8 + 4));
      const float y[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = y[j] - x[j];
    }
    const uint32_t w[4] = {kv[r].x, kv[r].y, kv[r].z, kv[r].w};
    const uint32_t o = sw128_chunk(t, c8, 64);
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float k0 = bf_lo(w[j]), k1 = bf_hi(w[j]);
      if (MODE == 0)
        split_bf2(k0 * __expf(-fmaxf(x[2 * j], -kSpanLimit)),
                  k1 * __expf(-fmaxf(x[2 * j + 1], -kSpanLimit)), hi[j], lo[j]);
      else
        split_bf2(k0 * __expf(x[2 * j]), k1 * __expf(x[2 * j + 1]), hi[j], lo[j]);
    }
    *reinterpret_cast<uint4*>(sm + off0 + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(sm + off0 + 16384 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (MODE == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        split_bf2(bf_lo(w[j]) * __expf(x[2 * j]), bf_hi(w[j]) * __expf(x[2 * j + 1]), hi[j], lo[j]);
      *reinterpret_cast<uint4*>(sm + off1 + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sm + off1 + 16384 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    kda_build_tc_kernel(const __grid_constant__ BuildParams p,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* sm = dsm_raw;
  Ctl& ctl = *reinterpret_cast<Ctl*>(sm + OFF_CTL);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.n_streams;
  if (p.ws->status != 0) return;  // the work list is not valid
  // the operand tiles need a 1024-aligned base (no room to pad one)
  if (sb & 1023u) {
    if (tid == 0) report(p.ws, HYPIC_ERR_CUDA, 299);
    return;
  }

  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(BAR(i), (i >= B_ITEMEMPTY0) ? kRingReaders : (i == B_WTREADY ? 2u : 1u));
    ctl.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t limit = p.spin_limit;

  // Bounded wait on completion number k of barrier i (parity k & 1); every role
  // leaves once any role gave up.
  auto wait_k = [&](int i, uint32_t k) -> bool {
    const uint32_t b = BAR(i), par = k & 1u;
    for (uint32_t n = 0; n < limit; ++n) {
      if (mbar_try(b, par)) return true;
      if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
    }
    if (atomicExch(&ctl.abort_flag, 1) == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, 200 + i);
    return false;
  };
  // the chunk scalars of chunk gg are published once per use of their slot
  auto wait_c = [&](uint32_t gg) { return wait_k(B_CREADY0 + (gg & 1u), gg >> 1); };
  const int n_items = p.n_items;
  auto ring_wait = [&](uint32_t k) { return wait_k(B_ITEMFULL0 + k % kRing, k / kRing); };
  auto ring_get = [&](uint32_t k) { return *reinterpret_cast<volatile int32_t*>(&ctl.ring[k % kRing]); };
  auto ring_release = [&](uint32_t k) { mbar_arrive(BAR(B_ITEMEMPTY0 + k % kRing)); };
  auto n_chunks = [&](int idx) { return idx < 0 ? 0 : (p.items[idx].len + kC - 1) / kC; };

  // =====================================================================
  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    // In order, sleeping on each input's barrier.  Window of chunk g:
    //   P_Q(g)   after W^T(g) and Qhat^T(g)     P_S(g)   after Shat^T(g), on U(g)
    //   Q update after R_Q(g) and Kn(g)         S update after R_S(g); then Kn is
    //                                           free (commit after both updates)
    //   G'(g+1)  after the images of g+1 (its tile held W(g), read into W^T(g)
    //            before W^T(g) was published)
    //   W(g+1)   after B(g+1) (the prep read G'(g+1) before publishing B)
    //   U(g+1)   after V(g+1); it restarts the P_S tile, whose R_S(g) the S update
    //            issued before it read
    // Every input of a window comes from work issued in earlier windows or
    // earlier in the same one, so the order cannot deadlock.
    if (lane == 0) {
      const uint32_t id_g = idesc_f16(128, 64) | ID_KK | ID_BF16;
      const uint32_t id_w = idesc_f16(128, 64) | ID_MM | ID_BF16;
      const uint32_t id_u = idesc_f16(128, 128) | ID_KM | ID_BF16;
      auto issue_G = [&]() {
        // M = 128 with the real rows in lanes 64..127: A starts 8 KB before each image
        const uint64_t ah = desc_sw128(sb + OFF_KP - 8192), al = desc_sw128(sb + OFF_KPL - 8192);
        const uint64_t bh = desc_sw128(sb + OFF_KM), bl = desc_sw128(sb + OFF_KML);
        mma8_ss<0, 2, 4, 6, 512, 514, 516, 518, 0, 2, 4, 6, 512, 514, 516, 518>(tmem + T_GW, ah, bh, id_g, 0u);
        mma8_ss<0, 2, 4, 6, 512, 514, 516, 518, 0, 2, 4, 6, 512, 514, 516, 518>(tmem + T_GW, ah, bl, id_g, 1u);
        mma8_ss<0, 2, 4, 6, 512, 514, 516, 518, 0, 2, 4, 6, 512, 514, 516, 518>(tmem + T_GW, al, bh, id_g, 1u);
        mma_commit(BAR(B_GDONE));
      };
      // W^T = (e^{c'} o K)^T B_W: A the MN-major view of the image (hi, then lo
      // 16 KB on), B_W hi and lo 8 KB apart; then the decayed U term V^T B_U,
      // starting the P_S tile
      auto issue_WU = [&](uint32_t gg) -> bool {
        if (!wait_k(B_BREADY, gg)) return false;
        tc_fence_after();
        const uint64_t a = desc_mn(sb + OFF_KP, 8192), b = desc_mn(sb + OFF_BWH, 8192);
        mma8_ss<0, 0, 128, 128, 256, 256, 384, 384, 0, 512, 128, 640, 256, 768, 384, 896>(
            tmem + T_GW, a, b, id_w, 0u);
        mma4_ss<1024, 1152, 1280, 1408, 0, 128, 256, 384>(tmem + T_GW, a, b, id_w);
        if (!wait_k(B_VFULL, gg)) return false;
        mma8_ss<0, 0, 128, 128, 256, 256, 384, 384, 0, 512, 128, 640, 256, 768, 384, 896>(
            tmem + T_PS, desc_mn(sb + OFF_V, 8192), desc_mn(sb + OFF_WT, 8192), id_w, 0u);
        mma_commit(BAR(B_WDONE));
        mma_commit(BAR(B_VEMPTY));
        return true;
      };
      auto issue_P = [&](uint32_t d, uint32_t xop, uint32_t acc0) {
        mma8_ss<0, 2, 4, 6, 1024, 1026, 1028, 1030, 0, 128, 256, 384, 512, 640, 768, 896>(
            tmem + d, desc_sw128(sb + xop), desc_mn(sb + OFF_WT, 8192), idesc_f16(128, 64) | ID_KM,
            acc0);
      };
      // X^T += R^T Kn: R^T hi/lo from tensor memory (hi of K step ks at column
      // 8 ks + 16 (ks / 2), lo 16 columns on) times Kn hi, then R^T hi times Kn lo
      auto issue_upd = [&](uint32_t dx, uint32_t rp) {
        const uint64_t b = desc_mn(sb + OFF_KN, 8192);
        mma8_ts<0, 16, 8, 24, 32, 48, 40, 56, 0, 0, 128, 128, 256, 256, 384, 384>(
            tmem + dx, tmem + rp, b, id_u);
        mma4_ts<0, 8, 32, 40, 1024, 1152, 1280, 1408>(tmem + dx, tmem + rp, b, id_u);
      };
      bool ok = true, pre = false;   // pre: G', W and U of chunk g were issued ahead
      uint32_t g = 0;
      for (uint32_t k = 0; ok; ++k) {
        if (!(ok = ring_wait(k))) break;
        const int idx = ring_get(k);
        ring_release(k);
        if (idx < 0) break;
        const int nc = n_chunks(idx);
        for (int c = 0; c < nc && ok; ++c, ++g) {
          bool has_next = (c + 1 < nc);
          if (!has_next) {   // the next item's first chunk, if it has one
            if (!(ok = ring_wait(k + 1))) break;
            has_next = n_chunks(ring_get(k + 1)) > 0;
          }
          if (!pre) {
            if (!(ok = wait_k(B_IMGREADY, g))) break;
            tc_fence_after();
            issue_G();
            if (!(ok = issue_WU(g))) break;
          }
          if (!(ok = wait_k(B_WTREADY, g) && wait_k(B_XQREADY, g))) break;
          tc_fence_after();
          issue_P(T_PQ, OFF_XQ, 0u);
          mma_commit(BAR(B_PQDONE));
          if (!(ok = wait_k(B_XSREADY, g))) break;
          tc_fence_after();
          issue_P(T_PS, OFF_XS, 1u);   // on top of the decayed U term
          mma_commit(BAR(B_PSDONE));
          if (!(ok = wait_k(B_RQREADY, g) && wait_k(B_KNREADY, g))) break;
          tc_fence_after();
          issue_upd(T_XQ, T_PQ);
          mma_commit(BAR(B_UQDONE));
          if (!(ok = wait_k(B_RSREADY, g))) break;
          tc_fence_after();
          issue_upd(T_XS, T_PS);
          mma_commit(BAR(B_USDONE));
          mma_commit(BAR(B_KNFREE));
          if (has_next) {
            if (!(ok = wait_k(B_IMGREADY, g + 1))) break;
            tc_fence_after();
            issue_G();
            if (!(ok = issue_WU(g + 1))) break;
          }
          pre = has_next;
        }
      }
      if (!ok) {
        mma_commit(BAR(B_DRAIN));
        mbar_wait(BAR(B_DRAIN), 0, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0, viss = 0, giss = 0;
      auto publish = [&](uint32_t k) -> bool {
        if (k >= kRing && !wait_k(B_ITEMEMPTY0 + k % kRing, k / kRing - 1)) return false;
        const uint32_t q = atomicAdd(&p.ws->queue, 1u);
        ctl.ring[k % kRing] = (q < static_cast<uint32_t>(n_items)) ? static_cast<int32_t>(q) : -1;
        mbar_arrive(BAR(B_ITEMFULL0 + k % kRing));
        return true;
      };
      ok = publish(0);
      for (uint32_t k = 0; ok; ++k) {
        const int idx = ctl.ring[k % kRing];
        if (idx < 0) break;
        if (!(ok = publish(k + 1))) break;   // one item ahead, for the prep's lookahead
        const WorkItem it = p.items[idx];
        const int nc = (it.len + kC - 1) / kC;
        const int s = it.unit % S;
        for (int c = 0; c < nc && ok; ++c, ++g) {
          const int32_t t0 = static_cast<int32_t>(it.tok_start + static_cast<int64_t>(c) * kC);
          // the gate tile, once the previous chunk's Kn has read c' (well before U
          // of the previous chunk frees V)
          if (g >= 1 && !(ok = wait_k(B_CPFREE, g - 1))) break;
          mbar_expect_tx(BAR(B_GFULL), 32768);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            tma_load_3d(sb + OFF_CP + 8192u * qq, &tm_g, BAR(B_GFULL), 32 * qq, s, t0);
          ++giss;
          if (g >= 1 && !(ok = wait_k(B_VEMPTY, g - 1))) break;
          mbar_expect_tx(BAR(B_VFULL), 16384);
          tma_load_3d(sb + OFF_V, &tm_v, BAR(B_VFULL), 0, s, t0);
          tma_load_3d(sb + OFF_V + 8192, &tm_v, BAR(B_VFULL), 64, s, t0);
          ++viss;
        }
      }
      if (!ok) {
        if (viss) mbar_wait(BAR(B_VFULL), (viss - 1) & 1u, kDrainLimit);
        if (giss) mbar_wait(BAR(B_GFULL), (giss - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ prep (256 threads)
    const int pt = tid - 64;                       // 0..255
    const int q = warp & 3;                        // TMEM lane quadrant
    const int hw = (warp >= 6) ? 1 : 0;            // this warp's half of a 64-column tile
    const int tl = q * 32 + lane;
    const __nv_bfloat16* __restrict__ kp = static_cast<const __nv_bfloat16*>(p.k);
    float* Lm = reinterpret_cast<float*>(sm + OFF_LIB);
    float* cp = reinterpret_cast<float*>(sm + OFF_CP);
    float* mt = reinterpret_cast<float*>(sm + OFF_MT);

    // The gates of chunk gg (their tile loaded by TMA): beta, the largest gate
    // m_t, the scans M and c', f = e^{M_n - M}, e^{c'_n}, the span flag; c' is
    // written over the gates (the swizzle repeats every eight tokens: element
    // (t, i) sits in 16-byte chunk (i / 4 mod 8) XOR (t mod 8) of row t).  Tokens
    // past the segment end take beta = 0 and gates 0.  Runs while the e^{-c'}
    // region is free (its last reader, W of the previous chunk, is done).  False
    // when the wait for the tile gave up.
    auto decay_chunk = [&](const WorkItem& it, int c, uint32_t gg) -> bool {
      const uint32_t slot = gg & 1u;
      const int64_t t0 = it.tok_start + static_cast<int64_t>(c) * kC;
      const int n = min(kC, it.len - c * kC);
      const int s = it.unit % S;
      float bv = 0.f;
      if (pt < n) bv = p.beta[(t0 + pt) * S + s];
      if (named_or(1, 256, (pt == 0) && !wait_k(B_GFULL, gg))) return false;
      {
        // warp w: tokens 8 (w - 2) .. + 7; lane l reads channels 4l .. 4l + 3
        const int w8 = (warp - 2) * 8;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int t = w8 + u;
          const float4 x = *reinterpret_cast<const float4*>(cp + cpi(t, 4 * lane));
          float m = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) mt[t] = (t < n) ? m : 0.f;
        }
        if (pt < kC) ctl.beta[slot][pt] = bv;
      }
      named_sync(1, 256);
      bool bad = false;
      if (pt < kD) {
        // c' of channel i = pt over the chunk, written over its gates: eight
        // tokens at a time, loaded together, scanned in registers, stored
        const int i = pt, ci = (i & 31) >> 2;
        float* col = cp + (i >> 5) * 2048 + (i & 3);
        float run = 0.f;
#pragma unroll 1
        for (int t8 = 0; t8 < kC; t8 += 8) {
          float x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] = col[(t8 + u) * 32 + ((ci ^ u) << 2)];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            run += (t8 + u < n) ? (x[u] - mt[t8 + u]) : 0.f;
            x[u] = run;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) col[(t8 + u) * 32 + ((ci ^ u) << 2)] = x[u];
        }
        ctl.gn[slot][i] = __expf(run);
        bad = run < -kSpanLimit;
      } else if (pt < kD + 32) {
        // M over token pairs (2 l, 2 l + 1), one warp
        const float m0 = mt[2 * lane], m1 = mt[2 * lane + 1];
        float sc = m0 + m1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += y;
        }
        const float Mn = __shfl_sync(0xffffffffu, sc, 31);
        ctl.ft[slot][2 * lane] = __expf(Mn - (sc - m1));
        ctl.ft[slot][2 * lane + 1] = __expf(Mn - sc);
        if (lane == 0) ctl.Mn[slot] = Mn;
      }
      bad = named_or(1, 256, bad);
      if (pt == 0) {
        ctl.bad[slot] = bad ? 1 : 0;
        mbar_arrive(BAR(B_CREADY0 + slot));
      }
      return true;
    };

    uint32_t g = 0;
    bool ok = true, have_c = false;   // have_c: the gates and keys of chunk g are in hand
    uint4 kv[4];                      // this thread's keys of the chunk (image items)
    for (uint32_t k = 0; ok; ++k) {
      if (named_or(1, 256, (pt == 0) && !ring_wait(k))) { ok = false; break; }
      const int idx = ring_get(k);
      named_sync(1, 256);
      if (pt == 0) ring_release(k);
      if (idx < 0) break;
      const WorkItem it = p.items[idx];
      const int nc = (it.len + kC - 1) / kC;
      const int s = it.unit % S;
      for (int c = 0; c < nc && ok; ++c, ++g) {
        const uint32_t slot = g & 1u;
        const int64_t t0 = it.tok_start + static_cast<int64_t>(c) * kC;
        const int n = min(kC, it.len - c * kC);
        if (!have_c) {
          load_keys(kp, t0, n, S, s, pt, kv);
          if (!(ok = decay_chunk(it, c, g))) break;
        }
        have_c = false;
        // (1) key images e^{-c'} o K and e^{c'} o K, once W of the previous chunk
        //     (the last reader of both regions) is done
        bool fail = (pt == 0) && g > 0 && !wait_k(B_WDONE, g - 1);
        if (named_or(1, 256, fail)) { ok = false; break; }
        key_images<0>(sm, OFF_KM, OFF_KP, cp, kv, pt);
        fence_proxy_async();
        named_sync(1, 256);
        if (pt == 0) mbar_arrive(BAR(B_IMGREADY));
        // (2) Kn, once the previous chunk's updates have read its region
        fail = (pt == 0) && g > 0 && !wait_k(B_KNFREE, g - 1);
        if (named_or(1, 256, fail)) { ok = false; break; }
        key_images<2>(sm, OFF_KN, 0, cp, kv, pt);
        fence_proxy_async();
        named_sync(1, 256);
        if (pt == 0) {
          mbar_arrive(BAR(B_KNREADY));
          mbar_arrive(BAR(B_CPFREE));   // c' read for the last time: the next gate tile may land
        }
        // (3) G' rows (lanes 64..127 = tokens) -> L = strictly-lower(beta_t G')
        fail = (pt == 0) && !wait_k(B_GDONE, g);
        if (named_or(1, 256, fail)) { ok = false; break; }
        tc_fence_after();
        if (q >= 2) {
          uint32_t r0[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + T_GW + 32 * hw, r0);
          tmem_wait_ld();
          const int t = tl - 64;
          const float bt = ctl.beta[slot][t];
          float* row = Lm + t * LROW + 32 * hw;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const int j = 32 * hw + jj;
            float4 v4;
            v4.x = (j + 0 < t) ? bt * __uint_as_float(r0[jj]) : 0.f;
            v4.y = (j + 1 < t) ? bt * __uint_as_float(r0[jj + 1]) : 0.f;
            v4.z = (j + 2 < t) ? bt * __uint_as_float(r0[jj + 2]) : 0.f;
            v4.w = (j + 3 < t) ? bt * __uint_as_float(r0[jj + 3]) : 0.f;
            *reinterpret_cast<float4*>(row + jj) = v4;
          }
        }
        tc_fence_before();
        named_sync(1, 256);
        // (4) Inv = (I + L)^-1 in place, 16x16 blocks: diagonal blocks by
        //     column solves, then the 2x2 recursion [[A^-1, 0], [-B^-1 C A^-1, B^-1]]
        {
          float x[16];
          const int rb = pt >> 4, j = pt & 15;
          if (pt < 64) {
            const float* Lb = Lm + (16 * rb) * LROW + 16 * rb;
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) x[ii] = (ii == j) ? 1.f : 0.f;
#pragma unroll
            for (int mm = 0; mm < 15; ++mm)
#pragma unroll
              for (int ii = mm + 1; ii < 16; ++ii) x[ii] = fmaf(-Lb[ii * LROW + mm], x[mm], x[ii]);
          }
          named_sync(1, 256);
          if (pt < 64) {
            float* Lb = Lm + (16 * rb) * LROW + 16 * rb;
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) Lb[ii * LROW + j] = x[ii];
          }
          named_sync(1, 256);
        }
        {
          float* Yt = reinterpret_cast<float*>(sm + OFF_YT);
          constexpr int YL = 36;
          if (pt < 64)
            smem_gemm<16, 16, 16, 1>(Yt, YL, Lm + 16 * LROW, LROW, Lm, LROW, 1.f, pt);
          else if (pt < 128)
            smem_gemm<16, 16, 16, 1>(Yt + 16 * YL, YL, Lm + 48 * LROW + 32, LROW,
                                     Lm + 32 * LROW + 32, LROW, 1.f, pt - 64);
          named_sync(1, 256);
          if (pt < 64)
            smem_gemm<16, 16, 16, 1>(Lm + 16 * LROW, LROW, Lm + 16 * LROW + 16, LROW, Yt, YL, -1.f, pt);
          else if (pt < 128)
            smem_gemm<16, 16, 16, 1>(Lm + 48 * LROW + 32, LROW, Lm + 48 * LROW + 48, LROW,
                                     Yt + 16 * YL, YL, -1.f, pt - 64);
          named_sync(1, 256);
          // product scratch: the W^T region, once P of the previous chunk has read
          // W^T there
          fail = (pt == 0) && g > 0 && !wait_k(B_PSDONE, g - 1);
          if (named_or(1, 256, fail)) { ok = false; break; }
          float* Ps = reinterpret_cast<float*>(sm + OFF_WT);
          gemm32_ksplit<true, false>(Yt, YL, Lm + 32 * LROW, LROW, Lm, LROW, 1.f, Ps, pt, 1);
          named_sync(1, 256);
          gemm32_ksplit<false, true>(Lm + 32 * LROW, LROW, Lm + 32 * LROW + 32, LROW, Yt, YL, -1.f,
                                     Ps, pt, 1);
          named_sync(1, 256);
        }
        // (5) B operands: B_W[j][t] = beta_j Inv[t][j] over L / Inv (read first),
        //     B_U = -f_j B_W[j][t] over the inverse's scratch; MN-major [64 j][64 t],
        //     bf16 hi + lo.  The epilogues write W^T(g) over B_U once W and U are done.
        {
          float vals[2][8];
          int jj[2], cc8[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int e = pt + 256 * r;
            jj[r] = e & 63;
            cc8[r] = e >> 6;
#pragma unroll
            for (int u = 0; u < 8; ++u) vals[r][u] = Lm[(8 * cc8[r] + u) * LROW + jj[r]];
          }
          named_sync(1, 256);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int j = jj[r];
            const float bj = ctl.beta[slot][j], nfj = -ctl.ft[slot][j];
            uint32_t wh[4], wl[4], uh[4], ul[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
              const float b0 = bj * vals[r][u], b1 = bj * vals[r][u + 1];
              split_bf2(b0, b1, wh[u >> 1], wl[u >> 1]);
              split_bf2(nfj * b0, nfj * b1, uh[u >> 1], ul[u >> 1]);
            }
            const uint32_t off = mn_chunk(cc8[r], j, 8192);
            *reinterpret_cast<uint4*>(sm + OFF_BWH + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            *reinterpret_cast<uint4*>(sm + OFF_BWL + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            *reinterpret_cast<uint4*>(sm + OFF_WT + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
            *reinterpret_cast<uint4*>(sm + OFF_WT + 8192 + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
          }
        }
        fence_proxy_async();
        named_sync(1, 256);
        if (pt == 0) mbar_arrive(BAR(B_BREADY));
        // (6) the keys and gates of the next chunk (this item's next chunk, or the
        //     first chunk of the next item), overlapping W, U and this chunk's
        //     state chain
        if (c + 1 < nc) {
          load_keys(kp, t0 + kC, min(kC, it.len - (c + 1) * kC), S, s, pt, kv);
          if (!(ok = decay_chunk(it, c + 1, g + 1))) break;
          have_c = true;
        } else {
          if (named_or(1, 256, (pt == 0) && !ring_wait(k + 1))) { ok = false; break; }
          const int nidx = ring_get(k + 1);
          if (n_chunks(nidx) > 0) {
            const WorkItem nx = p.items[nidx];
            load_keys(kp, nx.tok_start, min(kC, nx.len), S, nx.unit % S, pt, kv);
            if (!(ok = decay_chunk(nx, 0, g + 1))) break;
            have_c = true;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogues
    const bool is_q = warp < 14;
    const uint32_t nb = is_q ? 2 : 3;
    const int et = tid - (is_q ? 320 : 448);      // 0..127
    const int qd = warp & 3;
    const int ln = qd * 32 + lane;                 // TMEM lane = state column n
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t TX = is_q ? T_XQ : T_XS, TP = is_q ? T_PQ : T_PS;
    const uint32_t XOP = is_q ? OFF_XQ : OFF_XS;
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      if (named_or(nb, 128, (et == 0) && !ring_wait(k))) { ok = false; break; }
      const int idx = ring_get(k);
      named_sync(nb, 128);
      if (et == 0) ring_release(k);
      if (idx < 0) break;
      const WorkItem it = p.items[idx];
      const int nc = (it.len + kC - 1) / kC;
      const int64_t u = it.unit;
      float* __restrict__ outp = (is_q ? p.Qhat : p.S) + u * kD * kD;
      if (nc == 0) {
        for (int e = et; e < kD * kD; e += 128) outp[e] = (is_q && (e / kD) == (e % kD)) ? 1.f : 0.f;
        if (et == 0) {
          if (is_q) p.exp2[u] = 0; else p.log_T[u] = 0.f;
        }
        continue;
      }
      // ---- unit start: X^T = diag(e^{c'_n}) (Q) or 0 (S) pre-scaled for the
      //      first chunk; the state operand I or 0
      if (named_or(nb, 128, (et == 0) && !wait_c(g))) { ok = false; break; }
      bool bad = ctl.bad[g & 1u] != 0;
      double logM = ctl.Mn[g & 1u];
      {
        uint32_t r[32];
        const float d0 = ctl.gn[g & 1u][ln];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = (is_q && (b * 32 + e == ln)) ? __float_as_uint(d0) : 0u;
          tmem_st32(tmem + lane_off + TX + 32 * b, r);
        }
        tmem_wait_st();
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          uint4 w = make_uint4(0, 0, 0, 0);
          if (is_q && (c8 == (ln >> 3))) {
            const uint32_t one = 0x3C00u << (16 * (ln & 1));
            const int slotw = (ln & 7) >> 1;
            if (slotw == 0) w.x = one; else if (slotw == 1) w.y = one;
            else if (slotw == 2) w.z = one; else w.w = one;
          }
          *reinterpret_cast<uint4*>(sm + XOP + sw128_chunk(ln, c8, 128)) = w;
        }
        if (is_q && et == 0) {
          ctl.qmax[0] = __float_as_uint(1.f);
          ctl.qmax[1] = 0u;
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(nb, 128);
        if (et == 0) mbar_arrive(BAR(is_q ? B_XQREADY : B_XSREADY));
      }
      int exp2_acc = 0;
      for (int c = 0; c < nc && ok; ++c, ++g) {
        const bool last = (c == nc - 1);
        // ---- W^T (lane d, tokens 32 h .. 32 h + 31; h = 0 for Q, 1 for S) -> the
        //      W^T operand, fp16 MN-major [128 d][64 t], over the decayed-U operand
        //      (W and U are done)
        bool fail = (et == 0) && !wait_k(B_WDONE, g);
        if (named_or(nb, 128, fail)) { ok = false; break; }
        tc_fence_after();
        {
          const int h = is_q ? 0 : 1;
#pragma unroll 1
          for (int hb = 0; hb < 2; ++hb) {
            uint32_t r0[16];
            tmem_ld16(tmem + lane_off + T_GW + 32 * h + 16 * hb, r0);
            tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 2; ++c4) {
              const int o = c4 * 8;
              const uint4 w = make_uint4(pack_h2(__uint_as_float(r0[o]), __uint_as_float(r0[o + 1])),
                                         pack_h2(__uint_as_float(r0[o + 2]), __uint_as_float(r0[o + 3])),
                                         pack_h2(__uint_as_float(r0[o + 4]), __uint_as_float(r0[o + 5])),
                                         pack_h2(__uint_as_float(r0[o + 6]), __uint_as_float(r0[o + 7])));
              *reinterpret_cast<uint4*>(sm + OFF_WT + mn_chunk(4 * h + 2 * hb + c4, ln, 8192)) = w;
            }
          }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(nb, 128);
        if (et == 0) mbar_arrive(BAR(B_WTREADY));
        // ---- R epilogue: R^T = -P^T as bf16 hi/lo, written over P^T
        fail = (et == 0) && !wait_k(is_q ? B_PQDONE : B_PSDONE, g);
        if (named_or(nb, 128, fail)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pr[32];
          tmem_ld32(tmem + lane_off + TP + 32 * h, pr);
          tmem_wait_ld();
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            split_bf2(-__uint_as_float(pr[2 * e]), -__uint_as_float(pr[2 * e + 1]), hi[e], lo[e]);
          tmem_st16(tmem + lane_off + TP + 32 * h, hi);
          tmem_st16(tmem + lane_off + TP + 32 * h + 16, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        named_sync(nb, 128);
        if (et == 0) mbar_arrive(BAR(is_q ? B_RQREADY : B_RSREADY));
        // ---- state pass
        fail = (et == 0) && !wait_k(is_q ? B_UQDONE : B_USDONE, g);
        if (!last) fail = fail || ((et == 0) && !wait_c(g + 1));
        if (named_or(nb, 128, fail)) { ok = false; break; }
        tc_fence_after();
        if (!last) {
          const uint32_t ns = (g + 1) & 1u;
          float sc;
          if (is_q) {
            int e2;
            frexpf(__uint_as_float(ctl.qmax[c & 1]), &e2);
            const int sh = 1 - e2;
            exp2_acc -= sh;
            sc = ldexpf(1.f, sh);
            bad = bad || (ctl.bad[ns] != 0);
          } else {
            sc = __expf(ctl.Mn[ns]);
            logM += ctl.Mn[ns];
          }
          const float* gnx = ctl.gn[ns];
          float mloc = 0.f;
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + TX + 32 * b, r);
            tmem_wait_ld();
            // the state operand takes the scalar scale, tensor memory also the
            // next chunk's per-channel factor (column i = state row i)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float v = __uint_as_float(r[e]) * sc;
              mloc = fmaxf(mloc, fabsf(v));
              r[e] = __float_as_uint(v);
            }
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              const int o = c8 * 8;
              const uint4 w = make_uint4(pack_h2(__uint_as_float(r[o]), __uint_as_float(r[o + 1])),
                                         pack_h2(__uint_as_float(r[o + 2]), __uint_as_float(r[o + 3])),
                                         pack_h2(__uint_as_float(r[o + 4]), __uint_as_float(r[o + 5])),
                                         pack_h2(__uint_as_float(r[o + 6]), __uint_as_float(r[o + 7])));
              *reinterpret_cast<uint4*>(sm + XOP + sw128_chunk(ln, 4 * b + c8, 128)) = w;
            }
#pragma unroll
            for (int e4 = 0; e4 < 32; e4 += 4) {
              const float4 gv = *reinterpret_cast<const float4*>(gnx + 32 * b + e4);
              r[e4] = __float_as_uint(__uint_as_float(r[e4]) * gv.x);
              r[e4 + 1] = __float_as_uint(__uint_as_float(r[e4 + 1]) * gv.y);
              r[e4 + 2] = __float_as_uint(__uint_as_float(r[e4 + 2]) * gv.z);
              r[e4 + 3] = __float_as_uint(__uint_as_float(r[e4 + 3]) * gv.w);
            }
            tmem_st32(tmem + lane_off + TX + 32 * b, r);
          }
          tmem_wait_st();
          if (is_q) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
            if (et == 0) ctl.qmax[(c + 1) & 1] = 0u;
            named_sync(nb, 128);
            if (lane == 0) atomicMax(&ctl.qmax[(c + 1) & 1], __float_as_uint(mloc));
          }
          fence_proxy_async();
          tc_fence_before();
          named_sync(nb, 128);
          if (et == 0) mbar_arrive(BAR(is_q ? B_XQREADY : B_XSREADY));
        } else {
          // outputs: lane n holds column n of Qhat / S (rows i = 32 b + e)
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + TX + 32 * b, r);
            tmem_wait_ld();
            float* dst = outp + (32 * b) * kD + ln;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[e * kD] = __uint_as_float(r[e]);
          }
          tc_fence_before();
          named_sync(nb, 128);
          if (et == 0) {
            if (is_q) p.exp2[u] = bad ? kKdaRedo : exp2_acc;
            else p.log_T[u] = static_cast<float>(logM);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_build_kda_tc(const BuildParams& p, int n_sms, cudaStream_t st) {
  if (p.dk != kD || p.dv != kD) return launch_build_recurrence(p, HYPIC_BF16, st);
  CUtensorMap mv, mg;
  if (!make_token_map(&mv, p.v, p.n_tok, p.n_streams, kD) ||
      !make_gate_map(&mg, p.log_alpha, p.n_tok, p.n_streams, kD))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_build_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sms ? p.n_items : n_sms;
  kda_build_tc_kernel<<<grid, kThreads, SMEM_DYN, st>>>(p, mv, mg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // units whose decay span exceeded the single-reference bound, by the recurrence
  BuildParams r = p;
  r.redo_only = 1;
  return launch_build_recurrence(r, HYPIC_BF16, st);
}

}  // namespace hypic
