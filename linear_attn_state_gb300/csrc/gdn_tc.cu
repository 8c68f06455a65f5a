// Chunked gated-delta segment build on tcgen05 tensor cores (sm_103a).
//
// What it computes (youleyou.com HYPIC article, linear-layer paragraph): for
// every (segment, stream) unit the pair T_C = A_L ... A_1 and S(C|0), with
// A_t = alpha_t (I - beta_t k_t k_t^T) and S_t = A_t S_{t-1} + beta_t k_t v_t^T.
// T is carried factored, T = exp(log_T) 2^exp2 Qhat with Q = H_L ... H_1,
// H_t = I - beta_t k_t k_t^T (decay summed in log space, Q rescaled by exact
// powers of two), so long segments stay in fp32 range.
//
// Chunked WY/UT form, 64 tokens per chunk, c_i = within-chunk cumulative
// log-decay, Gamma_i = e^{c_i}, Gamma_n = e^{c_63}:
//   G   = K K^T,  L = strictly-lower(diag(beta) G),  Inv = (I + L)^-1
//   W   = Inv diag(beta) K
//   U   = (Inv o E) diag(beta) V,   E[t][j] = e^{c_t - c_j}   ((I + L o E)^-1 = Inv o E)
//   Q  <- Q + K^T R_Q,   R_Q = -W Qhat
//   S  <- S + K^T R_S,   R_S = diag(Gamma_n / Gamma_t) U - W Shat   (S pre-scaled by Gamma_n)
// Since (Gamma_n / Gamma_t) E[t][j] = e^{c_63 - c_j} = f_j, the decayed U term is
// Inv diag(beta f) V: it accumulates into the same tensor-memory tile as W Shat
// (with operand -f_j beta_j Inv[t][j]), and R_S = -(W Shat - Inv diag(beta f) V).
// The contractions run on tcgen05 (kind::f16, fp32 accumulators in tensor
// memory).  K and V enter as the bf16 they are given in: G, W, U and the state
// updates take bf16 operands, and the operands this kernel makes for them
// (beta Inv, beta Inv o E, R_Q, R_S) are split into bf16 hi + lo parts by
// truncation (two MMAs into one fp32 result; no conversion instructions).  The
// state operand of P = W Xhat and W^T are fp16 (11 significant bits).  The
// 64x64 unit-triangular inverse is an fp32 blocked solve on CUDA cores.
//
// The state is held transposed, X^T (tensor-memory lane = state column n, column
// = state row i), so that R^T can stay in tensor memory, written over P^T, and
// feed the update X^T += R^T K as the MMA's A operand.
//
// Warp roles (640 threads, one CTA per SM, persistent; each CTA takes the next
// item of the longest-first work list from a global queue when it needs one):
//   warp 0      MMA issuer (one thread) and tensor-memory owner
//   warp 1      TMA producer (one thread): K chunks into a 3-stage ring, V
//   warps 2-3   decay: beta and the cumulative log-decay of each chunk, ahead of the prep
//   warps 4-11  prep: L from G, the 64x64 inverse, the B operands of W and U,
//               W^T -> shared memory (two warps per SM sub-partition)
//   warps 12-15 Q-chain epilogue: R_Q, then the Q pass (rescale, Qhat)
//   warps 16-19 S-chain epilogue: R_S, then the S pass (pre-scale, Shat)
// The Q and S column halves of the state are independent chains, so the tensor
// pipe alternates between them while the next chunk's prep overlaps.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) X_Q^T  [128,256) X_S^T  [256,320) P_Q^T then R_Q^T hi/lo
//   [320,384) P_S^T (W Shat minus the decayed U term) then R_S^T hi/lo
//   [384,448) and [448,512) G (lanes 64..127) then W^T, by chunk parity
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "hypic_internal.h"
#include "tc_ptx.cuh"
#include "chunk_tc.cuh"

namespace hypic {
namespace {

using namespace tc;
using namespace chunk;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 640;

// ---- shared memory map (offsets from a 1024-aligned base) ----
constexpr uint32_t OFF_V = 0;            // V: [2 halves][64 t][64 d] bf16 SW128 (16 KB); its second
                                         // half is also the ignored rows the G MMA reads for stage 0
constexpr uint32_t OFF_K0 = 16384;       // K ring, 3 stages of 16 KB, same layout as V
constexpr uint32_t kKStages = 3;
constexpr uint32_t OFF_XQ = 65536;       // Qhat^T operand fp16, K-major [2 K blocks][128 n][64 i] (32 KB)
constexpr uint32_t OFF_XS = 98304;       // Shat^T operand (32 KB)
constexpr uint32_t OFF_WT = 131072;      // W^T operand fp16, MN-major [128 d][64 t] (16 KB)
constexpr uint32_t OFF_LIB = 147456;     // L / Inv fp32 [64][68] + inverse scratch, then B_W (24 KB)
constexpr uint32_t OFF_YT = OFF_LIB + 64 * 68 * 4;   // inverse scratch fp32 [32][36]
constexpr uint32_t OFF_BWH = OFF_LIB;            // beta Inv^T hi bf16, MN-major [64 j][64 t] (8 KB)
constexpr uint32_t OFF_BWL = OFF_LIB + 8192;     // ... lo
constexpr uint32_t OFF_BU0 = 172032;     // -(beta f Inv)^T hi, lo (decayed U term), 2 buffers
                                         // by chunk parity (16 KB each): read after the next prep began
constexpr uint32_t SMEM_END = OFF_BU0 + 32768;   // 204800
static_assert(OFF_YT + 32 * 36 * 4 <= SMEM_END, "inverse scratch overflows its region");
constexpr uint32_t SMEM_DYN = SMEM_END + 1024;
constexpr uint32_t LROW = 68;            // fp32 row stride of L / Inv

constexpr uint32_t T_XQ = 0, T_XS = 128, T_PQ = 256, T_PS = 320, T_GW0 = 384;   // G/W: 2 buffers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRing = 8;              // work-item ring between the TMA producer and the roles
constexpr uint32_t kRingReaders = 5;       // MMA, decay, prep, Q epilogue, S epilogue
constexpr uint32_t kDrainLimit = 1u << 20;  // suspending polls (~2 s)

// mbarrier slots
enum {
  B_KFULL0 = 0, B_KFULL1, B_KFULL2, B_VFULL, B_KEMPTY0, B_KEMPTY1, B_KEMPTY2, B_VEMPTY,
  B_KVREADY0, B_KVREADY1, B_KVREADY2, B_GDONE0, B_GDONE1, B_BREADY, B_WDONE, B_WTREADY, B_XQREADY,
  B_XSREADY, B_PQDONE, B_PSDONE,
  B_RQREADY, B_RSREADY, B_UQDONE, B_USDONE, B_DRAIN, B_ITEMFULL0,
  B_ITEMEMPTY0 = B_ITEMFULL0 + kRing, B_COUNT = B_ITEMEMPTY0 + kRing
};

struct Ctl {
  uint64_t bar[B_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
  float cs[kKStages][kC];     // ring like K: within-chunk cumulative log-decay c_t
  float ft[kKStages][kC];     // f_t = e^{c_63 - c_t} (<= 1)
  float beta[kKStages][kC];
  uint32_t qmax[2];     // max |Qhat| bits, alternating passes
  int32_t ring[kRing];  // work-list indices taken from the global queue, -1 = no more
  float conv_sum;       // decay role: decay sum of the chunk's first 32 tokens
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
  const int lane = tid & 31;
  const int S = p.n_streams;
  if (p.ws->status != 0) return;  // the work list is not valid

  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(BAR(i), (i >= B_ITEMEMPTY0) ? kRingReaders : 1u);
    ctl.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t limit = p.spin_limit;

  // Bounded wait on completion number k of barrier i (parity k & 1); checks the
  // CTA abort flag so that every role leaves once any role gave up.
  auto wait_k = [&](int i, uint32_t k) -> bool {
    const uint32_t b = BAR(i), par = k & 1u;
    for (uint32_t n = 0; n < limit; ++n) {
      if (mbar_try(b, par)) return true;
      if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
    }
    if (atomicExch(&ctl.abort_flag, 1) == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, 100 + i);
    return false;
  };

  // kv-ready completes once per chunk on the barrier of the chunk's ring
  // stage, so a consumer can never be two completions behind on one barrier
  auto wait_kv = [&](uint32_t gg) { return wait_k(B_KVREADY0 + gg % kKStages, gg / kKStages); };
  const int n_items = p.n_items;
  // Work items come from a global queue over the longest-first list (dynamic
  // LPT: a CTA takes the next item when it needs one).  The TMA producer takes
  // them and publishes the k-th in ring slot k % kRing; every role reads the
  // items in the same order.
  auto ring_wait = [&](uint32_t k) { return wait_k(B_ITEMFULL0 + k % kRing, k / kRing); };
  auto ring_get = [&](uint32_t k) { return *reinterpret_cast<volatile int32_t*>(&ctl.ring[k % kRing]); };
  auto ring_release = [&](uint32_t k) { mbar_arrive(BAR(B_ITEMEMPTY0 + k % kRing)); };
  auto n_chunks = [&](int idx) { return idx < 0 ? 0 : (p.items[idx].len + kC - 1) / kC; };

  // =====================================================================
  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    // In order, sleeping on each input's barrier (a suspending wait wakes as
    // the phase completes and takes no issue slots meanwhile).  Window of
    // chunk g:
    //   P_Q(g)   after W^T(g) and Qhat^T(g)      P_S(g)   after Shat^T(g)
    //   Q update after R_Q(g)                    S update after R_S(g); then K(g)
    //                                            is released (both updates read it)
    //   W(g+1)   after B(g+1) (and G(g+1), issued in an earlier window; the
    //            prep overwrites the W^T tile P_Q(g), P_S(g) read only after W(g+1))
    //   U(g+1)   after V(g+1) (it restarts the P_S tile, free once the S update
    //            of g was issued: the tensor pipe runs them in issue order)
    //   G(g+2)   after P_S(g) and K(g+2) (its G/W buffer held W^T(g), read into
    //            shared memory before W^T(g) was published)
    // Every input of a window depends only on work issued in earlier windows or
    // earlier in the same window, so the order cannot deadlock, and every
    // barrier is observed once per chunk, in order.
    if (lane == 0) {
      auto kaddr = [&](uint32_t gg) { return sb + OFF_K0 + (gg % kKStages) * 16384u; };
      auto gw = [&](uint32_t gg) { return tmem + T_GW0 + 64u * (gg & 1u); };
      auto issue_G = [&](uint32_t gg) {
        // M = 128 with the real rows in lanes 64..127: A starts 8 KB before the tile
        const uint32_t kb = kaddr(gg);
        mma8_ss<0, 2, 4, 6, 512, 514, 516, 518, 0, 2, 4, 6, 512, 514, 516, 518>(
            gw(gg), desc_sw128(kb - 8192), desc_sw128(kb), idesc_f16(128, 64) | ID_KK | ID_BF16, 0u);
        mma_commit(BAR(B_GDONE0 + (gg & 1u)));   // by parity: G can run two chunks ahead
      };
      // W^T = K^T B_W into the G/W buffer (A: MN-major view of the K tile; B_W
      // hi and lo 8 KB apart)
      auto issue_W = [&](uint32_t gg) {
        mma8_ss<0, 0, 128, 128, 256, 256, 384, 384, 0, 512, 128, 640, 256, 768, 384, 896>(
            gw(gg), desc_mn(kaddr(gg), 8192), desc_mn(sb + OFF_BWH, 8192),
            idesc_f16(128, 64) | ID_MM | ID_BF16, 0u);
        mma_commit(BAR(B_WDONE));
      };
      // the decayed U term V^T B_U starts the S-half P tile; V is then free
      auto issue_U = [&](uint32_t gg) {
        mma8_ss<0, 0, 128, 128, 256, 256, 384, 384, 0, 512, 128, 640, 256, 768, 384, 896>(
            tmem + T_PS, desc_mn(sb + OFF_V, 8192), desc_mn(sb + OFF_BU0 + (gg & 1u) * 16384u, 8192),
            idesc_f16(128, 64) | ID_MM | ID_BF16, 0u);
        mma_commit(BAR(B_VEMPTY));
      };
      // P^T(g) = Xhat^T W^T: A = Xhat^T (fp16, K-major, K blocks 16 KB apart), B = W^T
      auto issue_P = [&](uint32_t d, uint32_t xop, uint32_t acc0) {
        mma8_ss<0, 2, 4, 6, 1024, 1026, 1028, 1030, 0, 128, 256, 384, 512, 640, 768, 896>(
            tmem + d, desc_sw128(sb + xop), desc_mn(sb + OFF_WT, 8192), idesc_f16(128, 64) | ID_KM,
            acc0);
      };
      // X^T += R^T K: A = R^T hi, lo (bf16, tensor memory; hi of K step ks at
      // column 8 ks + 16 (ks / 2), lo 16 columns on), B = K (bf16, MN-major)
      auto issue_upd = [&](uint32_t dx, uint32_t rp, uint32_t kb) {
        mma8_ts<0, 16, 8, 24, 32, 48, 40, 56, 0, 0, 128, 128, 256, 256, 384, 384>(
            tmem + dx, tmem + rp, desc_mn(kb, 8192), idesc_f16(128, 128) | ID_KM | ID_BF16);
      };
      bool ok = true, pre = false;   // pre: G, W and U of chunk g were issued ahead
      uint32_t g = 0, g_issued = 0;  // G issued for chunks below g_issued
      auto want_G = [&](uint32_t gg) -> bool {   // issue G(gg) if not yet issued
        if (g_issued > gg) return true;
        if (!wait_kv(gg)) return false;
        tc_fence_after();
        issue_G(gg);
        g_issued = gg + 1;
        return true;
      };
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
          // does chunk g+2 exist (known without looking past the next item)?
          bool has_next2 = (c + 2 < nc);
          if (!has_next2) {
            if (c + 2 == nc && !(ok = ring_wait(k + 1))) break;
            const int nn = n_chunks(ring_get(k + 1));
            has_next2 = (c + 2 == nc) ? (nn > 0) : (nn > 1);
          }
          const uint32_t kb = kaddr(g);
          const uint32_t n1 = g + 1;
          if (!pre) {  // G, W and U of this chunk (nothing in flight before them)
            if (!(ok = want_G(g))) break;
            if (has_next && !(ok = want_G(n1))) break;
            if (!(ok = wait_k(B_BREADY, g))) break;
            tc_fence_after();
            issue_W(g);
            if (!(ok = wait_k(B_VFULL, g))) break;
            issue_U(g);
          }
          if (!(ok = wait_k(B_WTREADY, g) && wait_k(B_XQREADY, g))) break;
          tc_fence_after();
          issue_P(T_PQ, OFF_XQ, 0u);
          mma_commit(BAR(B_PQDONE));
          if (!(ok = wait_k(B_XSREADY, g))) break;
          tc_fence_after();
          issue_P(T_PS, OFF_XS, 1u);   // on top of the decayed U term
          mma_commit(BAR(B_PSDONE));
          // G(g+2) now, so that it is done before the prep of g+2 starts
          if (has_next2 && !(ok = want_G(g + 2))) break;
          if (!(ok = wait_k(B_RQREADY, g))) break;
          tc_fence_after();
          issue_upd(T_XQ, T_PQ, kb);
          mma_commit(BAR(B_UQDONE));
          if (!(ok = wait_k(B_RSREADY, g))) break;
          tc_fence_after();
          issue_upd(T_XS, T_PS, kb);
          mma_commit(BAR(B_USDONE));
          mma_commit(BAR(B_KEMPTY0 + g % kKStages));
          if (has_next) {
            if (!(ok = want_G(n1) && wait_k(B_BREADY, n1))) break;
            tc_fence_after();
            issue_W(n1);
            if (!(ok = wait_k(B_VFULL, n1))) break;
            issue_U(n1);
          }
          pre = has_next;
        }
      }
      if (!ok) {
        // let every MMA issued so far land before tensor memory is released
        mma_commit(BAR(B_DRAIN));
        mbar_wait(BAR(B_DRAIN), 0, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0;
      uint32_t kiss[kKStages] = {0, 0, 0}, viss = 0;   // loads issued per barrier
      // K runs one chunk ahead of V: the next chunk's K is issued before this
      // chunk's V waits for the decayed U term of the previous chunk to free V
      uint32_t gk = 0;   // K issued for the chunks below gk
      auto load_k = [&](uint32_t gg, int sk, int32_t tk) -> bool {
        const uint32_t st = gg % kKStages;
        if (gg >= kKStages && !wait_k(B_KEMPTY0 + st, gg / kKStages - 1)) return false;
        const uint32_t kb = sb + OFF_K0 + st * 16384u;
        mbar_expect_tx(BAR(B_KFULL0 + st), 16384);
        tma_load_3d(kb, &tm_k, BAR(B_KFULL0 + st), 0, sk, tk);
        tma_load_3d(kb + 8192, &tm_k, BAR(B_KFULL0 + st), 64, sk, tk);
        ++kiss[st];
        gk = gg + 1;
        return true;
      };
      // take the next work item from the global queue into ring slot k
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
        if (!(ok = publish(k + 1))) break;   // one item ahead, for the roles that look ahead
        const WorkItem it = p.items[idx];
        const int nc = (it.len + kC - 1) / kC;
        const int s = it.unit % S;
        for (int c = 0; c < nc && ok; ++c, ++g) {
          const int32_t t0 = static_cast<int32_t>(it.tok_start + static_cast<int64_t>(c) * kC);
          if (gk == g && !(ok = load_k(g, s, t0))) break;
          // the next chunk's K: this item's next chunk, or the first chunk of the
          // next item (published one item ahead; an empty next item ends the lookahead)
          if (c + 1 < nc) {
            if (!(ok = load_k(g + 1, s, t0 + kC))) break;
          } else {
            const int nidx = ctl.ring[(k + 1) % kRing];
            if (nidx >= 0 && n_chunks(nidx) > 0) {
              const WorkItem nx = p.items[nidx];
              if (!(ok = load_k(g + 1, nx.unit % S, static_cast<int32_t>(nx.tok_start)))) break;
            }
          }
          if (g >= 1 && !(ok = wait_k(B_VEMPTY, g - 1))) break;
          mbar_expect_tx(BAR(B_VFULL), 16384);
          tma_load_3d(sb + OFF_V, &tm_v, BAR(B_VFULL), 0, s, t0);
          tma_load_3d(sb + OFF_V + 8192, &tm_v, BAR(B_VFULL), 64, s, t0);
          ++viss;
        }
      }
      if (!ok) {
        // drain the copies this thread issued (waiting on an already observed
        // completion returns at once)
        for (uint32_t st = 0; st < kKStages; ++st)
          if (kiss[st]) mbar_wait(BAR(B_KFULL0 + st), (kiss[st] - 1) & 1u, kDrainLimit);
        if (viss) mbar_wait(BAR(B_VFULL), (viss - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ prep (256 threads)
    const int pt = tid - 128;                      // 0..255
    const int q = warp & 3;                        // TMEM lane quadrant
    const int tl = q * 32 + lane;                  // TMEM lane of this thread
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      if (named_or(1, 256, (pt == 0) && !ring_wait(k))) { ok = false; break; }
      const int idx = ring_get(k);
      named_sync(1, 256);
      if (pt == 0) ring_release(k);
      if (idx < 0) break;
      const int nc = n_chunks(idx);
      for (int c = 0; c < nc && ok; ++c, ++g) {
        const uint32_t slot = g % kKStages, slot2 = g & 1u;
        bool fail;
        // (3) G rows (lanes 64..127 = tokens 0..63) -> L = strictly-lower(beta_t G)
        fail = (pt == 0) && !wait_k(B_GDONE0 + slot2, g >> 1);
        fail = named_or(1, 256, fail);
        if (fail) { ok = false; break; }
        tc_fence_after();
        float* Lm = reinterpret_cast<float*>(sm + OFF_LIB);
        if (q >= 2) {
          // warps of quadrants 2-3 (lanes 64..127 = tokens); one half of the columns each
          const int h = (warp >= 8) ? 1 : 0;
          uint32_t r0[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + T_GW0 + 64 * slot2 + 32 * h, r0);
          tmem_wait_ld();
          const int t = tl - 64;
          const float bt = ctl.beta[slot][t];
          float* row = Lm + t * LROW + 32 * h;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const int j = 32 * h + jj;
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
        // (4) Inv = (I + L)^-1 in place, 16x16 blocks.
        //  (a) diagonal blocks by column solves (threads 0..63)
        {
          float x[16];
          const int rb = pt >> 4, j = pt & 15;
          if (pt < 64) {
            // column j of the block inverse, column-oriented: once x_m is final
            // it updates every later row, so the 15 updates of a step are
            // independent (dependency depth 15 instead of 120)
            const float* Lb = Lm + (16 * rb) * LROW + 16 * rb;
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m)
#pragma unroll
              for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-Lb[i * LROW + m], x[m], x[i]);
          }
          named_sync(1, 256);
          if (pt < 64) {
            float* Lb = Lm + (16 * rb) * LROW + 16 * rb;
#pragma unroll
            for (int i = 0; i < 16; ++i) Lb[i * LROW + j] = x[i];
          }
          named_sync(1, 256);
        }
        //  (b) 2x2 recursion: with A = rows/cols 0..31 and B = 32..63,
        //      (I+L)^-1 = [[A^-1, 0], [-B^-1 C A^-1, B^-1]], and likewise for the
        //      16x16 halves of A and B.  Temporaries in the scratch region.
        {
          float* Yt = reinterpret_cast<float*>(sm + OFF_YT);   // [32][36] fp32
          constexpr int YL = 36;
          // level 1: Y0 = L[16:32,0:16] D0^-1,  Y1 = L[48:64,32:48] D2^-1
          if (pt < 64)
            smem_gemm<16, 16, 16, 1>(Yt, YL, Lm + 16 * LROW, LROW, Lm, LROW, 1.f, pt);
          else if (pt < 128)
            smem_gemm<16, 16, 16, 1>(Yt + 16 * YL, YL, Lm + 48 * LROW + 32, LROW,
                                     Lm + 32 * LROW + 32, LROW, 1.f, pt - 64);
          named_sync(1, 256);
          //          X10 = -D1^-1 Y0 -> L[16:32,0:16];  X32 = -D3^-1 Y1 -> L[48:64,32:48]
          if (pt < 64)
            smem_gemm<16, 16, 16, 1>(Lm + 16 * LROW, LROW, Lm + 16 * LROW + 16, LROW, Yt, YL, -1.f, pt);
          else if (pt < 128)
            smem_gemm<16, 16, 16, 1>(Lm + 48 * LROW + 32, LROW, Lm + 48 * LROW + 48, LROW,
                                     Yt + 16 * YL, YL, -1.f, pt - 64);
          named_sync(1, 256);
          // level 2: Y = C A^-1 (C = L[32:64,0:32]), then L[32:64,0:32] = -B^-1 Y.
          // Scratch: the decayed-U operand buffer of this chunk's parity, whose
          // previous contents were consumed before this chunk's G completed and
          // which is rewritten only at step (5).
          float* Ps = reinterpret_cast<float*>(sm + OFF_BU0 + slot2 * 16384u);
          gemm32_ksplit<true, false>(Yt, YL, Lm + 32 * LROW, LROW, Lm, LROW, 1.f, Ps, pt, 1);
          named_sync(1, 256);
          gemm32_ksplit<false, true>(Lm + 32 * LROW, LROW, Lm + 32 * LROW + 32, LROW, Yt, YL, -1.f,
                                     Ps, pt, 1);
          named_sync(1, 256);
        }
        // (5) B operands: B_W[j][t] = beta_j Inv[t][j] and B_U = -f_j B_W[j][t];
        //     MN-major [64 j][64 t], bf16 hi + lo.  Read first, then overwrite.
        {
          float vals[2][8];
          int jj[2], cc8[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int e = pt + 256 * r;        // 512 chunks: (j, 8 consecutive t)
            jj[r] = e & 63;                    // consecutive lanes: consecutive j (no conflicts)
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
            uint8_t* bu = sm + OFF_BU0 + slot2 * 16384u;
            *reinterpret_cast<uint4*>(bu + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
            *reinterpret_cast<uint4*>(bu + 8192 + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
          }
        }
        fence_proxy_async();
        named_sync(1, 256);
        if (pt == 0) mbar_arrive(BAR(B_BREADY));
        // (6) W^T (lane d, column t) -> W^T operand, MN-major [128 d][64 t]
        fail = (pt == 0) && !wait_k(B_WDONE, g);
        fail = named_or(1, 256, fail);
        if (fail) { ok = false; break; }
        tc_fence_after();
        {
          const int h = (warp >= 8) ? 1 : 0;   // this warp's half of the 64 token columns
          uint32_t r0[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + T_GW0 + 64 * slot2 + 32 * h, r0);
          tmem_wait_ld();
          const int d = tl;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c8 = 4 * h + c4;
            uint4 w;
            const uint32_t* src = r0;
            const int o = c4 * 8;
            w.x = pack_h2(__uint_as_float(src[o]), __uint_as_float(src[o + 1]));
            w.y = pack_h2(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3]));
            w.z = pack_h2(__uint_as_float(src[o + 4]), __uint_as_float(src[o + 5]));
            w.w = pack_h2(__uint_as_float(src[o + 6]), __uint_as_float(src[o + 7]));
            *reinterpret_cast<uint4*>(sm + OFF_WT + mn_chunk(c8, d, 8192)) = w;
          }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(1, 256);
        if (pt == 0) mbar_arrive(BAR(B_WTREADY));
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogues
    const bool is_q = warp < 16;
    const uint32_t nb = is_q ? 2 : 3;              // named barrier id
    const int et = tid - (is_q ? 384 : 512);       // 0..127
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
        // identity pair
        for (int e = et; e < kD * kD; e += 128) outp[e] = (is_q && (e / kD) == (e % kD)) ? 1.f : 0.f;
        if (et == 0) {
          if (is_q) p.exp2[u] = 0; else p.log_T[u] = 0.f;
        }
        continue;
      }
      // ---- unit start: X^T = [I | 0], Xhat^T likewise (row n of the K-major operand)
      {
        uint32_t r[32];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = (is_q && (b * 32 + e == ln)) ? 0x3f800000u : 0u;
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
      double logG = 0.0;
      for (int c = 0; c < nc && ok; ++c, ++g) {
        const uint32_t slot = g % kKStages;
        const bool last = (c == nc - 1);
        // ---- R epilogue
        bool fail = (et == 0) && !wait_k(is_q ? B_PQDONE : B_PSDONE, g);
        fail = named_or(nb, 128, fail);
        if (fail) { ok = false; break; }
        tc_fence_after();
        const float c_last = ctl.cs[slot][kC - 1];
        // R^T (lane n, tokens t) in bf16 hi/lo, written over P^T: tokens 0..31
        // (read first) into columns [0,32), then tokens 32..63 into [32,64)
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
        // the S pass pre-scales by the next chunk's decay: wait for it
        float gnext = 0.f;
        const bool has_next_global = !is_q && !last;
        tc_fence_before();
        fail = false;
        if (!is_q && has_next_global) fail = (et == 0) && !wait_kv(g + 1);
        fail = named_or(nb, 128, fail);
        if (fail) { ok = false; break; }
        if (!is_q && has_next_global) gnext = ctl.cs[(g + 1) % kKStages][kC - 1];
        if (et == 0) mbar_arrive(BAR(is_q ? B_RQREADY : B_RSREADY));
        if (!is_q && et == 0) logG += static_cast<double>(c_last);
        // ---- state pass
        fail = (et == 0) && !wait_k(is_q ? B_UQDONE : B_USDONE, g);
        fail = named_or(nb, 128, fail);
        if (fail) { ok = false; break; }
        tc_fence_after();
        if (!last) {
          float sc;
          if (is_q) {
            int e2;
            frexpf(__uint_as_float(ctl.qmax[c & 1]), &e2);
            const int sh = 1 - e2;
            exp2_acc -= sh;
            sc = ldexpf(1.f, sh);
          } else {
            sc = __expf(gnext);
          }
          float mloc = 0.f;
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + TX + 32 * b, r);
            tmem_wait_ld();
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
          // outputs: lane n holds column n of Qhat / S (rows i = 32 b + e); a
          // warp's 32 lanes store 32 consecutive floats of one row
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
            if (is_q) p.exp2[u] = exp2_acc;
            else p.log_T[u] = static_cast<float>(logG);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ decay (warps 2-3)
    // Each chunk's beta and within-chunk cumulative log-decay, ahead of the
    // prep; published with kv-ready once the chunk's K has landed.  Tokens past
    // the segment end get beta = 0 and log-decay 0: with beta_t = 0 row t of L
    // and of Inv is the identity's and W, U and R vanish there, so whatever the
    // K and V tiles hold in those rows (finite inputs, or the zero fill past the
    // end of the tensor) contributes exactly nothing.  Thread ct owns token ct.
    const int ct = tid - 64;                       // 0..63
    uint32_t g = 0;
    bool ok = true;
    auto load_bg = [&](int idx, int c, float& b, float& gg) {
      b = gg = 0.f;
      if (idx < 0) return;
      const WorkItem it = p.items[idx];
      const int64_t t0 = it.tok_start + static_cast<int64_t>(c) * kC;
      const int n = min(kC, it.len - c * kC);
      const int s = it.unit % S;
      if (ct < n) {
        b = p.beta[(t0 + ct) * S + s];
        gg = p.log_alpha[(t0 + ct) * S + s];
      }
    };
    // beta and log-decay are loaded one chunk ahead: the next chunk of the item,
    // else the first chunk of the next item
    float nb = 0.f, ng = 0.f;
    bool have_next = false;
    for (uint32_t k = 0; ok; ++k) {
      if (named_or(4, 64, (ct == 0) && !ring_wait(k))) { ok = false; break; }
      const int idx = ring_get(k);
      named_sync(4, 64);
      if (ct == 0) ring_release(k);
      if (idx < 0) break;
      const int nc = n_chunks(idx);
      for (int c = 0; c < nc && ok; ++c, ++g) {
        const uint32_t slot = g % kKStages;
        if (!have_next) load_bg(idx, c, nb, ng);
        const float bcur = nb, gcur = ng;
        have_next = false;
        if (c + 1 < nc) {
          load_bg(idx, c + 1, nb, ng);
          have_next = true;
        } else {
          if (named_or(4, 64, (ct == 0) && !ring_wait(k + 1))) { ok = false; break; }
          const int nidx = ring_get(k + 1);
          if (n_chunks(nidx) > 0) {
            load_bg(nidx, 0, nb, ng);
            have_next = true;
          }
        }
        bool fail = (ct == 0) && !wait_k(B_KFULL0 + slot, g / kKStages);
        if (named_or(4, 64, fail)) { ok = false; break; }
        float sc = gcur;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += y;
        }
        if (ct == 31) ctl.conv_sum = sc;
        named_sync(4, 64);
        if (ct >= 32) sc += ctl.conv_sum;
        ctl.cs[slot][ct] = sc;
        ctl.beta[slot][ct] = bcur;
        {
          const float clast = __shfl_sync(0xffffffffu, sc, 31);   // warp 15: token 63
          named_sync(4, 64);
          if (ct == 63) ctl.conv_sum = clast;
          named_sync(4, 64);
          const float c63 = ctl.conv_sum;
          ctl.ft[slot][ct] = __expf(c63 - sc);
        }
        named_sync(4, 64);
        if (ct == 0) mbar_arrive(BAR(B_KVREADY0 + slot));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_build_gdn_tc(const BuildParams& p, int n_sms, cudaStream_t st) {
  if (p.dk != kD || p.dv != kD) return launch_build_recurrence(p, HYPIC_BF16, st);
  CUtensorMap mk, mv;
  if (!make_token_map(&mk, p.k, p.n_tok, p.n_streams, kD) ||
      !make_token_map(&mv, p.v, p.n_tok, p.n_streams, kD))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gdn_build_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_DYN));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sms ? p.n_items : n_sms;
  gdn_build_tc_kernel<<<grid, kThreads, SMEM_DYN, st>>>(p, mk, mv);
  return cudaGetLastError();
}


}  // namespace hypic
