// Segment build for the decay-only families on tcgen05 tensor cores (sm_103a).
//
// What it computes (youleyou.com HYPIC article, linear-layer paragraph: the
// cached pair is the segment's transition product and its zero-start state):
// for a unit (segment, stream) with body tokens t = 0..L-1,
//   RetNet (scalar gamma):  T_C = gamma^L I,           S = sum_t gamma^{L-1-t} k_t v_t^T
//   GLA (per key channel):  T_C = diag(e^{G_L}),       S = sum_t diag(e^{G_L - G_{t+1}}) k_t v_t^T
//   plain linear attention: T_C = I,                   S = sum_t k_t v_t^T
//   Mamba2-style (per-token scalar): T_C = e^{G_L} I,  S = sum_t e^{G_L - G_{t+1}} k_t v_t^T
// with G_t the running sum of the log-decays g over the first t tokens; the
// decay of token t is the product of the decays of the tokens after it.  So S
// is one contraction, S = (W o K)^T V, W[t][i] = exp(sum_{t' > t} g[t'][i])
// (or gamma^{L-1-t}, or 1; the per-token scalar gate is the same for every i).
//
// Per unit the 64-token chunks are taken in reverse order, so the suffix sum
// of g is a running value: within a chunk it is accumulated in fp32 (64 terms),
// across chunks in fp64 (it also gives log T for GLA).  A = W o K is formed in
// fp32 and split into bf16 hi + lo by truncation (16 significant bits); V is
// the bf16 input, exact.  Two MMAs per 16 tokens (hi, lo) accumulate S^T in
// fp32 tensor memory: D[n][i] += sum_t V[t][n] A[t][i].
//
// Warp roles (512 threads, one CTA per SM, persistent over a strided share of
// the longest-first work list):
//   warp 0      MMA issuer (one thread) and tensor-memory owner
//   warp 1      TMA producer: K (plain rows), V (128-byte swizzle, the MMA's
//               MN-major layout) and, for GLA, g of each chunk into a ring of
//               4 stages (2 with g); for the per-token gate, a 4-stream x 64-
//               token box of g into a small ring of its own
//   warps 4-11  builders: A = W o K -> the MN-major A operand (double-buffered),
//               log T.  The weights first: GLA, thread (i, h) runs the suffix
//               sums of key channel i over the token half h and writes the
//               weights over the g tile; one weight per token (RetNet, Mamba2-
//               style, plain), a 64-entry table.  Then each thread scales 8
//               channels x 1 token per step (16-byte loads of K and the weights,
//               16-byte stores of the hi and lo parts)
//   warps 12-15 epilogue: S from tensor memory (double-buffered, held transposed:
//               lane = column n) to HBM, one coalesced row segment per warp store
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "hypic_internal.h"
#include "tc_ptx.cuh"

namespace hypic {
namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 512;

// shared memory (offsets from a 1024-aligned base): A hi | lo (16 KB each),
// 2 buffers, then the input ring: per stage V 16 KB | K 16 KB, 4 stages; the
// builders' half sums (1 KB); the per-token gate ring (4 stages x 1 KB: 64
// tokens x 4 streams fp32).  With a per-channel decay (GLA) V has a ring of its
// own (3 stages of 16 KB, freed by the MMA) and K with the 32 KB gate tile
// another (2 stages of 48 KB, freed by the builders once A is formed), so the
// next chunks' K and gates load while the MMA still reads V.
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_STAGE = 65536;
constexpr uint32_t ST_V = 0, ST_K = 16384, ST_G = 32768;
template <int KIND> struct Ring {
  static constexpr uint32_t kStages = (KIND == 2) ? 3 : 4;        // V stages (with K unless GLA)
  static constexpr uint32_t kBytes = (KIND == 2) ? 16384 : 32768;
  static constexpr uint32_t kRegion = (KIND == 2) ? 49152 + 2 * 49152 : 131072;
};
constexpr uint32_t OFF_KG = OFF_STAGE + 49152;    // GLA: K | g stages of 48 KB
constexpr uint32_t kKGBytes = 49152;
constexpr uint32_t OFF_G4 = OFF_STAGE + 131072 + 1024;
constexpr uint32_t kG4Bytes = 64 * 4 * 4;
template <int KIND>
constexpr uint32_t smem_dyn() {
  return OFF_STAGE + Ring<KIND>::kRegion + 1024 + (KIND == 4 ? 4 * kG4Bytes : 0) + 1024;
}
constexpr uint32_t kTmemCols = 256;        // 2 D buffers of 128 columns
constexpr uint32_t kDrainLimit = 1u << 20;

enum {
  D_FULL0 = 0, D_EMPTY0 = 4, D_AREADY0 = 8, D_AFREE0 = 10, D_DFULL0 = 12, D_DFREE0 = 14,
  D_DRAIN = 16, D_KGFULL0 = 17, D_KGEMPTY0 = 19, D_COUNT = 21
};

struct DCtl {
  uint64_t bar[D_COUNT];
  uint32_t tmem_base;
  int32_t abort_flag;
};

static_assert(smem_dyn<2>() + sizeof(DCtl) <= 232448 && smem_dyn<4>() + sizeof(DCtl) <= 232448,
              "shared memory over the per-CTA limit");

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
// byte offset of the 2-byte element (mn, k) of an MN-major SW128 tile whose
// 64-wide MN atoms are `lbo` bytes apart (K rows 128 bytes apart)
__device__ __forceinline__ uint32_t mn_elem(uint32_t mn, uint32_t k, uint32_t lbo) {
  return (mn >> 6) * lbo + (k >> 3) * 1024u + (k & 7u) * 128u +
         ((((mn >> 3) & 7u) ^ (k & 7u)) << 4) + ((mn & 7u) << 1);
}
}  // namespace

// KIND: 1 scalar decay (RetNet), 2 per-channel decay (GLA), 3 none, 4 per-token
// scalar decay (Mamba2-style; n_streams a multiple of 4)
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    decay_build_tc_kernel(const __grid_constant__ BuildParams p,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ DCtl ctl;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.n_streams;
  if (p.ws->status != 0) return;  // the work list is not valid

  auto BAR = [&](int i) { return smem_u32(&ctl.bar[i]); };
  if (tid == 0) {
    for (int i = 0; i < D_COUNT; ++i) mbar_init(BAR(i), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    if (KIND == 2 || KIND == 4) prefetch_tmap(&tm_g);
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
    if (atomicExch(&ctl.abort_flag, 1) == 0) report(p.ws, HYPIC_ERR_DEVICE_TIMEOUT, 300 + i);
    return false;
  };
  using R = Ring<KIND>;
  const int n_items = p.n_items;
  const int first = blockIdx.x, stride = gridDim.x;
  auto n_chunks = [&](int ix) { return (p.items[ix].len + kC - 1) / kC; };

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_f16(128, 128) | (1u << 15) | (1u << 16) | (1u << 7) | (1u << 10);
      bool ok = true;
      uint32_t g = 0, un = 0;   // chunks and non-empty units of this CTA so far
      for (int ix = first; ix < n_items && ok; ix += stride) {
        const int nc = n_chunks(ix);
        if (nc == 0) continue;
        const uint32_t db = un & 1u;
        // the epilogue has drained this D buffer (unit un - 2)
        if (un >= 2 && !(ok = wait_k(D_DFREE0 + db, (un >> 1) - 1))) break;
        tc_fence_after();
        for (int c = 0; c < nc && ok; ++c, ++g) {
          const uint32_t st = g % R::kStages, ab = g & 1u;
          if (!(ok = wait_k(D_FULL0 + st, g / R::kStages) && wait_k(D_AREADY0 + ab, g >> 1))) break;
          tc_fence_after();
          const uint32_t va = sb + OFF_STAGE + st * R::kBytes + ST_V;   // V (its own ring for GLA)
          const uint32_t aa = sb + OFF_A + ab * 32768u;
          // D[n][i] += sum_t V[t][n] A[t][i]: S transposed, so that the
          // epilogue's warps store rows of S with consecutive lanes
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t av = desc_mn(va + ks * 2048, 8192);
            mma_f16(tmem + 128 * db, av, desc_mn(aa + ks * 2048, 8192), id, (c > 0 || ks > 0));
            mma_f16(tmem + 128 * db, av, desc_mn(aa + 16384 + ks * 2048, 8192), id, 1);
          }
          mma_commit(BAR(D_EMPTY0 + st));
          mma_commit(BAR(D_AFREE0 + ab));
        }
        if (!ok) break;
        mma_commit(BAR(D_DFULL0 + db));
        ++un;
      }
      if (!ok) {
        mma_commit(BAR(D_DRAIN));
        mbar_wait(BAR(D_DRAIN), 0, kDrainLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0, iss[4] = {0, 0, 0, 0}, kgiss[2] = {0, 0};
      const uint32_t bytes = (KIND == 2 ? 16384u : 32768u) + (KIND == 4 ? kG4Bytes : 0u);
      for (int ix = first; ix < n_items && ok; ix += stride) {
        const WorkItem it = p.items[ix];
        const int nc = (it.len + kC - 1) / kC;
        const int s = it.unit % S;
        for (int c = nc - 1; c >= 0 && ok; --c, ++g) {   // chunks in reverse
          const uint32_t st = g % R::kStages;
          const int32_t t0 = static_cast<int32_t>(it.tok_start + static_cast<int64_t>(c) * kC);
          if constexpr (KIND == 2) {
            // K and the gate tile, once the builders are done with the stage
            const uint32_t sk = g & 1u, kb = sb + OFF_KG + sk * kKGBytes, kbar = BAR(D_KGFULL0 + sk);
            if (g >= 2 && !(ok = wait_k(D_KGEMPTY0 + sk, (g >> 1) - 1))) break;
            mbar_expect_tx(kbar, 16384u + 32768u);
            tma_load_3d(kb, &tm_k, kbar, 0, s, t0);
            tma_load_3d(kb + 16384, &tm_g, kbar, 0, s, t0);
            ++kgiss[sk];
          }
          if (g >= R::kStages && !(ok = wait_k(D_EMPTY0 + st, g / R::kStages - 1))) break;
          const uint32_t base = sb + OFF_STAGE + st * R::kBytes, bar = BAR(D_FULL0 + st);
          mbar_expect_tx(bar, bytes);
          tma_load_3d(base + ST_V, &tm_v, bar, 0, s, t0);
          tma_load_3d(base + ST_V + 8192, &tm_v, bar, 64, s, t0);
          if (KIND != 2) tma_load_3d(base + ST_K, &tm_k, bar, 0, s, t0);
          if (KIND == 4) tma_load_3d(sb + OFF_G4 + st * kG4Bytes, &tm_g, bar, 0, s >> 2, t0);
          ++iss[st];
        }
      }
      if (!ok) {
        for (uint32_t st = 0; st < R::kStages; ++st)
          if (iss[st]) mbar_wait(BAR(D_FULL0 + st), (iss[st] - 1) & 1u, kDrainLimit);
        for (uint32_t sk = 0; sk < 2; ++sk)
          if (kgiss[sk]) mbar_wait(BAR(D_KGFULL0 + sk), (kgiss[sk] - 1) & 1u, kDrainLimit);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------- builders
    const int bt = tid - 128;          // 0..255
    float* hsum = reinterpret_cast<float*>(sm + OFF_STAGE + R::kRegion);  // [2][128]
    bool ok = true;
    uint32_t g = 0;
    for (int ix = first; ix < n_items && ok; ix += stride) {
      const WorkItem it = p.items[ix];
      const int nc = (it.len + kC - 1) / kC;
      const int s = it.unit % S;
      double run = 0.0;            // sum of g over the tokens after the current chunk
      float lg = 0.f;
      if (KIND == 1) lg = p.log_alpha[s];
      for (int c = nc - 1; c >= 0 && ok; --c, ++g) {
        const uint32_t st = g % R::kStages, ab = g & 1u;
        // the chunk's K (and gates): the input stage, or for GLA the K | g stage
        bool fail = (bt == 0) && !(((KIND == 2) ? wait_k(D_KGFULL0 + (g & 1u), g >> 1)
                                                : wait_k(D_FULL0 + st, g / R::kStages)) &&
                                   (g < 2 || wait_k(D_AFREE0 + ab, (g >> 1) - 1)));
        if (named_or(1, 256, fail)) { ok = false; break; }
        const int n = min(kC, it.len - c * kC);   // valid tokens of this chunk
        const uint8_t* stg = (KIND == 2) ? sm + OFF_KG + (g & 1u) * kKGBytes
                                         : sm + OFF_STAGE + st * R::kBytes + ST_K;
        const __nv_bfloat16* kt = reinterpret_cast<const __nv_bfloat16*>(stg);
        uint8_t* ah = sm + OFF_A + ab * 32768u;
        uint8_t* al = ah + 16384;
        if (KIND == 2) {
          // (1) the weights, in place of g: w[t][i] = exp(sum of g[.][i] over the
          //     tokens after t in the unit); thread (i, h): key channel i, token
          //     half h (t in [32 h, 32 h + 32))
          const int i = bt & 127, h = bt >> 7;
          float* gw = reinterpret_cast<float*>(sm + OFF_KG + (g & 1u) * kKGBytes + 16384);
          const int tb = 32 * h;
          // the thread's 32 gates, read once into registers; both halves' sums:
          // the later half's starts the earlier half's suffix
          float gr[32];
          float sh = 0.f;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            gr[u] = (tb + u < n) ? gw[(tb + u) * kD + i] : 0.f;
            sh += gr[u];
          }
          hsum[h * kD + i] = sh;
          named_sync(1, 256);
          float loc = (h == 0) ? hsum[kD + i] : 0.f;   // g summed over the later tokens
          const float ctot = hsum[i] + hsum[kD + i];
          const float runf = static_cast<float>(run);
#pragma unroll
          for (int u = 31; u >= 0; --u) {
            gw[(tb + u) * kD + i] = (tb + u < n) ? __expf(runf + loc) : 0.f;
            loc += gr[u];
          }
          run += static_cast<double>(ctot);
          named_sync(1, 256);
          // (2) A = w o K, 8 channels x 1 token per step (as below, with the
          //     weights read from the tile)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pq = bt + 256 * j;
            const int t = pq >> 4, c8 = pq & 15;
            const uint4 kr = *reinterpret_cast<const uint4*>(kt + t * kD + 8 * c8);
            const float4 w0 = *reinterpret_cast<const float4*>(gw + t * kD + 8 * c8);
            const float4 w1 = *reinterpret_cast<const float4*>(gw + t * kD + 8 * c8 + 4);
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a0 = wv[2 * e] * __uint_as_float(kw[e] << 16);
              const float a1 = wv[2 * e + 1] * __uint_as_float(kw[e] & 0xFFFF0000u);
              const uint32_t u0 = __float_as_uint(a0), u1 = __float_as_uint(a1);
              hi[e] = __byte_perm(u0, u1, 0x7632);
              const float r0 = a0 - __uint_as_float(u0 & 0xFFFF0000u);
              const float r1 = a1 - __uint_as_float(u1 & 0xFFFF0000u);
              lo[e] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            }
            const uint32_t off = mn_elem(8 * c8, t, 8192);
            *reinterpret_cast<uint4*>(ah + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(al + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        } else {
          // (1) the chunk's 64 token weights (one per token: the decay after it)
          float* wt = hsum;   // [64]
          if (bt < kC) {
            const int t = bt;
            float w = 0.f;
            if (KIND == 1) w = (t < n) ? __expf(lg * static_cast<float>(it.len - 1 - (c * kC + t))) : 0.f;
            if (KIND == 3) w = (t < n) ? 1.f : 0.f;
            if (KIND == 4) {
              // g of the later tokens of the chunk: reverse scan over the two warps
              const float* g4 = reinterpret_cast<const float*>(sm + OFF_G4 + st * kG4Bytes);
              const float gv = (t < n) ? g4[t * 4 + (s & 3)] : 0.f;
              float x = gv;   // sum over tokens t..31 of this warp (inclusive)
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, x, o);
                if (lane + o < 32) x += y;
              }
              if (t == 32) hsum[64] = x;            // tokens 32..63
              asm volatile("bar.sync 5, 64;" ::: "memory");
              const float upper = (t < 32) ? hsum[64] : 0.f;
              const float later = x - gv + upper;   // tokens after t
              w = (t < n) ? __expf(static_cast<float>(run) + later) : 0.f;
              const float ctot = __shfl_sync(0xffffffffu, x, 0) + upper;   // whole chunk (warp 0)
              asm volatile("bar.sync 5, 64;" ::: "memory");
              if (t == 0) hsum[65] = ctot;
            }
            wt[t] = w;
          }
          named_sync(1, 256);
          if (KIND == 4) run += static_cast<double>(hsum[65]);
          // (2) A = w o K, 8 channels x 1 token per step: one 16-byte load of K,
          //     one 16-byte store each of the hi and lo parts (MN-major chunk)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pq = bt + 256 * j;
            const int t = pq >> 4, c8 = pq & 15;
            const float w = wt[t];
            const uint4 kr = *reinterpret_cast<const uint4*>(kt + t * kD + 8 * c8);
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a0 = w * __uint_as_float(kw[e] << 16);
              const float a1 = w * __uint_as_float(kw[e] & 0xFFFF0000u);
              const uint32_t u0 = __float_as_uint(a0), u1 = __float_as_uint(a1);
              hi[e] = __byte_perm(u0, u1, 0x7632);
              const float r0 = a0 - __uint_as_float(u0 & 0xFFFF0000u);
              const float r1 = a1 - __uint_as_float(u1 & 0xFFFF0000u);
              lo[e] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            }
            const uint32_t off = mn_elem(8 * c8, t, 8192);
            *reinterpret_cast<uint4*>(ah + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(al + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async();
        named_sync(1, 256);
        if (bt == 0) {
          mbar_arrive(BAR(D_AREADY0 + ab));
          if (KIND == 2) mbar_arrive(BAR(D_KGEMPTY0 + (g & 1u)));   // K and gates read
        }
      }
      if (!ok) break;
      const int64_t u = it.unit;
      if (KIND == 2 && bt < kD) p.log_T[u * kD + bt] = static_cast<float>(run);   // per channel
      if (bt == 0) {
        if (KIND == 1)
          p.log_T[u] = static_cast<float>(static_cast<double>(it.len) * static_cast<double>(lg));
        if (KIND == 3) p.log_T[u] = 0.f;
        if (KIND == 4) p.log_T[u] = static_cast<float>(run);
      }
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;   // TMEM lane = S column n
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    uint32_t un = 0;
    for (int ix = first; ix < n_items && ok; ix += stride) {
      const WorkItem it = p.items[ix];
      float* dst = p.S + static_cast<int64_t>(it.unit) * kD * kD + row;   // column n of S
      if (it.len == 0) {   // empty body: S = 0
        for (int e = 0; e < kD; ++e) dst[e * kD] = 0.f;
        continue;
      }
      const uint32_t db = un & 1u;
      bool fail = (row == 0) && !wait_k(D_DFULL0 + db, un >> 1);
      if (named_or(2, 128, fail)) { ok = false; break; }
      tc_fence_after();
      // rows i = 32 b + e: a warp's 32 lanes store 32 consecutive floats of row i
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + 128 * db + 32 * b, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[(32 * b + e) * kD] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      named_sync(2, 128);
      if (row == 0) mbar_arrive(BAR(D_DFREE0 + db));
      ++un;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_d() {
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

// 3-D map over [n_tok][n_streams][128]; box = inner x 1 stream x 64 tokens
bool make_map3(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams, bool f32,
               uint32_t inner, bool swizzle) {
  auto fn = encode_fn_d();
  if (!fn) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(n_streams),
                        static_cast<cuuint64_t>(n_tok)};
  cuuint64_t strides[2] = {kD * es, kD * es * static_cast<cuuint64_t>(n_streams)};
  cuuint32_t box[3] = {inner, 1u, static_cast<cuuint32_t>(kC)};
  cuuint32_t ones[3] = {1u, 1u, 1u};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-token gates [n_tok][n_streams] fp32 as [n_tok][n_streams / 4][4]; box =
// 4 streams x 64 tokens (the x coordinate is always 0: 16-byte aligned)
bool make_map_g4(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams) {
  auto fn = encode_fn_d();
  if (!fn) return false;
  cuuint64_t dims[3] = {4u, static_cast<cuuint64_t>(n_streams / 4), static_cast<cuuint64_t>(n_tok)};
  cuuint64_t strides[2] = {16u, 4u * static_cast<cuuint64_t>(n_streams)};
  cuuint32_t box[3] = {4u, 1u, static_cast<cuuint32_t>(kC)};
  cuuint32_t ones[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch_decay_kind(const BuildParams& p, int n_sms, cudaStream_t st) {
  CUtensorMap mk, mv, mg;
  if (!make_map3(&mk, p.k, p.n_tok, p.n_streams, false, kD, false) ||
      !make_map3(&mv, p.v, p.n_tok, p.n_streams, false, 64, true))
    return cudaErrorInvalidValue;
  mg = mk;   // unused without a per-token gate
  if (KIND == 2 && !make_map3(&mg, p.log_alpha, p.n_tok, p.n_streams, true, kD, false))
    return cudaErrorInvalidValue;
  if (KIND == 4 && !make_map_g4(&mg, p.log_alpha, p.n_tok, p.n_streams)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decay_build_tc_kernel<KIND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_dyn<KIND>()));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sms ? p.n_items : n_sms;
  decay_build_tc_kernel<KIND><<<grid, kThreads, smem_dyn<KIND>(), st>>>(p, mk, mv, mg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_build_decay(const BuildParams& p, int n_sms, cudaStream_t st) {
  if (p.dk != kD || p.dv != kD) return launch_build_recurrence(p, HYPIC_BF16, st);
  switch (p.kind) {
    case HYPIC_SCALAR_DECAY: return launch_decay_kind<1>(p, n_sms, st);
    case HYPIC_DIAG_DECAY: return launch_decay_kind<2>(p, n_sms, st);
    case HYPIC_TOKEN_DECAY:
      // the gate box needs 16-byte rows of 4 streams and a 16-byte aligned base
      if (p.n_streams % 4 != 0 || (reinterpret_cast<uintptr_t>(p.log_alpha) & 15u) != 0)
        return launch_build_recurrence(p, HYPIC_BF16, st);
      return launch_decay_kind<4>(p, n_sms, st);
    default: return launch_decay_kind<3>(p, n_sms, st);
  }
}

}  // namespace hypic
