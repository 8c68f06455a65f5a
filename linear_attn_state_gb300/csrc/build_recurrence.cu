// Work-list preparation and the fp32 token-recurrence segment build.
//
// prepare: derives the longest-body-first (LPT) work list of (segment, stream)
// items from the device offsets (youleyou.com HYPIC article, segment-
// parallelism paragraph: LPT balancing of cold segments).
//
// build_recurrence: one CTA per (segment, stream) unit runs the per-token
// recurrence of the unit's body exactly as defined (linear-layer paragraph:
// T_C is the ordered product of the per-token transitions, S(C|0) the final
// state from zero), in fp32 on CUDA cores.  Used for fp32 inputs (where fp16
// tensor-core operands would round the inputs), for dk = dv = 64, for KDA, and
// for Mamba2-style heads whose stream count is not a multiple of 4.
// Thread n owns column n of X = [Q | S] (dk rows), so every token is a local
// dot product and a rank-1 update with the key broadcast from shared memory:
//   x <- alpha x + k (b vval - alpha beta (k . x)),  vval = 0 on Q columns.
// KDA (the gated delta rule with a per-key-channel gate a = e^g, decay first):
//   y = a o x,  x <- y + k (beta vval - beta (k . y));
// its Q columns take the gate relative to the token's largest one,
// e^(g - max g) <= 1, and log T sums the largest gates, so the factored T =
// e^(log T) 2^exp2 Qhat keeps the slowest channel's scale.
#include <cuda_bf16.h>

#include "hypic_internal.h"

namespace hypic {

// Offsets are read as off[i] - tok_base (a slice of a longer offsets array when
// a build covers a group of segments); unit indices start at seg_off * n_streams.
// Body cost of segment j: its length minus the seam window (an invalid range
// costs 0 and is reported by its own thread).
__device__ __forceinline__ int64_t body_cost(const int64_t* __restrict__ off, int32_t j,
                                             int32_t seam_w, int64_t n_tok, int64_t tok_base) {
  const int64_t a = off[j] - tok_base, b = off[j + 1] - tok_base;
  const int64_t L = (b >= a && a >= 0 && b <= n_tok) ? (b - a) : 0;
  return L - (L < seam_w ? L : seam_w);
}

constexpr int kPrepThreads = 256;
constexpr int kPrepStreams = 32;   // streams whose items one block writes

// Thread i ranks segment i: rank = number of segments ordered before it by
// (-cost, segment).  The costs are read in tiles of kPrepThreads through
// shared memory (one coalesced load per tile), so the n_seg^2 comparisons run
// from shared memory.  With index_order the rank is the segment index.
__global__ void __launch_bounds__(kPrepThreads)
    build_prepare_kernel(const int64_t* __restrict__ off, int32_t n_seg, int32_t seam_w,
                         int32_t n_streams, int64_t n_tok, int64_t tok_base, int32_t seg_off,
                         int32_t index_order, WorkItem* __restrict__ items, WsHeader* ws) {
  __shared__ int64_t cost_s[kPrepThreads];
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  const bool mine = i < n_seg;
  int64_t a = 0, cost = 0, w = 0;
  if (mine) {
    a = off[i] - tok_base;
    const int64_t b = off[i + 1] - tok_base;
    bool ok = (b >= a) && (a >= 0) && (b <= n_tok);
    if (i == 0 && a != 0) ok = false;
    if (i == n_seg - 1 && b != n_tok) ok = false;
    const int64_t L = ok ? (b - a) : 0;
    w = L < seam_w ? L : seam_w;
    cost = L - w;
    if (!ok) report(ws, HYPIC_ERR_OFFSETS, 1);
  }
  int32_t rank = 0;
  for (int32_t j0 = 0; j0 < n_seg && !index_order; j0 += kPrepThreads) {
    __syncthreads();
    const int32_t j = j0 + static_cast<int32_t>(threadIdx.x);
    if (j < n_seg) cost_s[threadIdx.x] = body_cost(off, j, seam_w, n_tok, tok_base);
    __syncthreads();
    const int32_t nj = min(kPrepThreads, n_seg - j0);
    if (mine)
      for (int32_t jj = 0; jj < nj; ++jj) {
        const int64_t cj = cost_s[jj];
        rank += (cj > cost) || (cj == cost && j0 + jj < i);
      }
  }
  if (!mine) return;
  if (index_order) rank = i;
  // this block's slices of the streams (blockIdx.y, striding by gridDim.y):
  // the rank is recomputed per block, so the items of a segment are written by
  // many threads at once
  for (int64_t s0 = static_cast<int64_t>(blockIdx.y) * kPrepStreams; s0 < n_streams;
       s0 += static_cast<int64_t>(gridDim.y) * kPrepStreams) {
    const int32_t s1 = static_cast<int32_t>(min(static_cast<int64_t>(n_streams), s0 + kPrepStreams));
    for (int32_t s = static_cast<int32_t>(s0); s < s1; ++s) {
      WorkItem it;
      it.tok_start = a + w;
      it.len = static_cast<int32_t>(cost);
      it.unit = (seg_off + i) * n_streams + s;
      items[static_cast<int64_t>(rank) * n_streams + s] = it;
    }
  }
}

cudaError_t launch_build_prepare(const int64_t* d_offsets, int32_t n_seg, int32_t seam_w,
                                 int32_t n_streams, int64_t n_tok, int64_t tok_base,
                                 int32_t seg_off, bool index_order, WorkItem* items, WsHeader* ws,
                                 cudaStream_t st) {
  if (n_seg == 0) return cudaSuccess;
  const int64_t slices = (static_cast<int64_t>(n_streams) + kPrepStreams - 1) / kPrepStreams;
  const dim3 grid((n_seg + kPrepThreads - 1) / kPrepThreads,
                  static_cast<unsigned>(slices < 65535 ? slices : 65535));
  build_prepare_kernel<<<grid, kPrepThreads, 0, st>>>(
      d_offsets, n_seg, seam_w, n_streams, n_tok, tok_base, seg_off, index_order ? 1 : 0, items,
      ws);
  return cudaGetLastError();
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

constexpr int kTile = 16;  // tokens staged in shared memory per step

// KIND: 0 gdn, 1 scalar, 2 diag, 3 none, 4 per-token scalar, 5 kda.
// Threads: DK + DV (gdn, kda: Q and S columns) or DV.
template <typename Tin, int DK, int DV, int KIND>
__global__ void __launch_bounds__((KIND == 0 || KIND == 5) ? DK + DV : DV)
    build_recurrence_kernel(BuildParams p) {
  constexpr bool kMat = (KIND == 0 || KIND == 5);   // Q columns: a matrix transition
  constexpr int NT = kMat ? DK + DV : DV;
  __shared__ __align__(16) float k_s[kTile][DK];
  __shared__ __align__(16) float v_s[kTile][DV];
  __shared__ __align__(16) float a_s[kTile][(KIND == 2 || KIND == 5) ? DK : 1];
  __shared__ __align__(16) float aq_s[kTile][KIND == 5 ? DK : 1];   // gate / largest gate
  __shared__ float alpha_s[kTile];
  __shared__ float beta_s[kTile];
  __shared__ float g_s[kTile];
  __shared__ float red_s[32];

  if (p.ws->status != 0) return;  // the work list is not valid
  const WorkItem it = p.items[blockIdx.x];
  if (p.redo_only && p.exp2[it.unit] != kKdaRedo) return;
  const int tid = threadIdx.x;
  const int S = p.n_streams;
  const int stream = it.unit % S;
  const Tin* __restrict__ kp = static_cast<const Tin*>(p.k);
  const Tin* __restrict__ vp = static_cast<const Tin*>(p.v);

  const bool is_q = kMat && (tid < DK);
  const int col = kMat ? (is_q ? tid : tid - DK) : tid;

  // the column, in pairs of rows: the token loops run as packed two-wide fp32
  // operations (the same operations, in the same order, as scalar ones)
  float2 xp[DK / 2];
  auto X = [&](int i) -> float& { return (i & 1) ? xp[i >> 1].y : xp[i >> 1].x; };
#pragma unroll
  for (int i = 0; i < DK; ++i) X(i) = (is_q && i == col) ? 1.f : 0.f;
  int exp2_acc = 0;
  double logG = 0.0;  // thread 0 (gdn, token, kda) or thread i<DK (diag)

  float gamma_alpha = 1.f;
  if (KIND == 1) gamma_alpha = expf(p.log_alpha[stream]);

  for (int t0 = 0; t0 < it.len; t0 += kTile) {
    const int nt = min(kTile, it.len - t0);
    __syncthreads();
    for (int e = tid; e < kTile * DK; e += NT) {
      const int tt = e / DK, i = e % DK;
      float kv = 0.f;
      if (tt < nt) kv = to_f(kp[((it.tok_start + t0 + tt) * S + stream) * DK + i]);
      k_s[tt][i] = kv;
      if (KIND == 2 || KIND == 5) {
        float ga = 0.f;
        if (tt < nt) ga = p.log_alpha[((it.tok_start + t0 + tt) * S + stream) * DK + i];
        a_s[tt][i] = (KIND == 2) ? expf(ga) : ga;   // kda: the log-gate, exponentiated below
        // per-channel log-decay sum kept by thread i (threads >= DK hold none)
      }
    }
    for (int e = tid; e < kTile * DV; e += NT) {
      const int tt = e / DV, j = e % DV;
      v_s[tt][j] = (tt < nt) ? to_f(vp[((it.tok_start + t0 + tt) * S + stream) * DV + j]) : 0.f;
    }
    if ((KIND == 0 || KIND == 4 || KIND == 5) && tid < kTile) {
      float b = 0.f, g = 0.f;
      if (tid < nt) {
        if (KIND != 4) b = p.beta[(it.tok_start + t0 + tid) * S + stream];
        if (KIND != 5) g = p.log_alpha[(it.tok_start + t0 + tid) * S + stream];
      }
      beta_s[tid] = b;
      g_s[tid] = g;
      alpha_s[tid] = expf(g);
    }
    __syncthreads();
    if (KIND == 5) {
      // the token's largest log-gate (0 for padding rows), then both gates
      if (tid < kTile) {
        float m = -INFINITY;
        for (int i = 0; i < DK; ++i) m = fmaxf(m, a_s[tid][i]);
        g_s[tid] = (tid < nt) ? m : 0.f;
      }
      __syncthreads();
      for (int e = tid; e < kTile * DK; e += NT) {
        const int tt = e / DK, i = e % DK;
        const float ga = a_s[tt][i];
        aq_s[tt][i] = expf(ga - g_s[tt]);
        a_s[tt][i] = expf(ga);
      }
      __syncthreads();
    }
    if (KIND == 2 && tid < DK) {
      for (int tt = 0; tt < nt; ++tt)
        logG += static_cast<double>(p.log_alpha[((it.tok_start + t0 + tt) * S + stream) * DK + tid]);
    }
    if ((KIND == 0 || KIND == 4 || KIND == 5) && tid == 0)
      for (int tt = 0; tt < nt; ++tt) logG += static_cast<double>(g_s[tt]);

    for (int tt = 0; tt < nt; ++tt) {
      const float vval = is_q ? 0.f : v_s[tt][col];
      if (KIND == 0) {
        float2 ua = make_float2(0.f, 0.f), ub = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&k_s[tt][i]);
          ua = __ffma2_rn(make_float2(kk.x, kk.y), xp[i >> 1], ua);
          ub = __ffma2_rn(make_float2(kk.z, kk.w), xp[(i >> 1) + 1], ub);
        }
        const float u = (ua.x + ua.y) + (ub.x + ub.y);
        // Q columns carry the ungated product (the decay lives in log_T)
        const float al = is_q ? 1.f : alpha_s[tt], be = beta_s[tt];
        const float c = be * vval - al * be * u;
        const float2 al2 = make_float2(al, al), c2 = make_float2(c, c);
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&k_s[tt][i]);
          xp[i >> 1] = __ffma2_rn(al2, xp[i >> 1], __fmul2_rn(make_float2(kk.x, kk.y), c2));
          xp[(i >> 1) + 1] =
              __ffma2_rn(al2, xp[(i >> 1) + 1], __fmul2_rn(make_float2(kk.z, kk.w), c2));
        }
      } else if (KIND == 5) {
        // y = a o x (decay first), then the delta-rule correction along k
        const float* __restrict__ ar = is_q ? aq_s[tt] : a_s[tt];
        float2 ua = make_float2(0.f, 0.f), ub = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&k_s[tt][i]);
          const float4 aa = *reinterpret_cast<const float4*>(&ar[i]);
          xp[i >> 1] = __fmul2_rn(xp[i >> 1], make_float2(aa.x, aa.y));
          xp[(i >> 1) + 1] = __fmul2_rn(xp[(i >> 1) + 1], make_float2(aa.z, aa.w));
          ua = __ffma2_rn(make_float2(kk.x, kk.y), xp[i >> 1], ua);
          ub = __ffma2_rn(make_float2(kk.z, kk.w), xp[(i >> 1) + 1], ub);
        }
        const float be = beta_s[tt];
        const float c = be * vval - be * ((ua.x + ua.y) + (ub.x + ub.y));
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&k_s[tt][i]);
          xp[i >> 1] = __ffma2_rn(make_float2(kk.x, kk.y), c2, xp[i >> 1]);
          xp[(i >> 1) + 1] = __ffma2_rn(make_float2(kk.z, kk.w), c2, xp[(i >> 1) + 1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < DK; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&k_s[tt][i]);
          float a0 = 1.f, a1 = 1.f, a2 = 1.f, a3 = 1.f;
          if (KIND == 1) a0 = a1 = a2 = a3 = gamma_alpha;
          if (KIND == 4) a0 = a1 = a2 = a3 = alpha_s[tt];
          if (KIND == 2) {
            const float4 aa = *reinterpret_cast<const float4*>(&a_s[tt][i]);
            a0 = aa.x; a1 = aa.y; a2 = aa.z; a3 = aa.w;
          }
          const float2 v2 = make_float2(vval, vval);
          xp[i >> 1] = __ffma2_rn(make_float2(a0, a1), xp[i >> 1],
                                  __fmul2_rn(make_float2(kk.x, kk.y), v2));
          xp[(i >> 1) + 1] = __ffma2_rn(make_float2(a2, a3), xp[(i >> 1) + 1],
                                        __fmul2_rn(make_float2(kk.z, kk.w), v2));
        }
      }
    }

    // Power-of-two rescale of Q (gdn, kda) every 64 tokens: Q = 2^exp2 * Qhat.
    if (kMat && (((t0 + kTile) & 63) == 0 || t0 + kTile >= it.len)) {
      float m = 0.f;
      if (is_q) {
#pragma unroll
        for (int i = 0; i < DK; ++i) m = fmaxf(m, fabsf(X(i)));
      }
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      __syncthreads();
      if ((tid & 31) == 0) red_s[tid >> 5] = m;
      __syncthreads();
      float mm = 0.f;
      for (int w = 0; w < (DK + 31) / 32; ++w) mm = fmaxf(mm, red_s[w]);
      if (mm > 0.f && (mm < 1.f || mm >= 2.f)) {
        int e2;
        frexpf(mm, &e2);          // mm = f * 2^e2, f in [0.5, 1)
        const int sh = 1 - e2;    // mm * 2^sh in [1, 2)
        exp2_acc -= sh;
        if (is_q) {
#pragma unroll
          for (int i = 0; i < DK; ++i) X(i) = ldexpf(X(i), sh);
        }
      }
    }
  }

  const int64_t u = it.unit;
  if (kMat) {
    if (is_q) {
#pragma unroll
      for (int i = 0; i < DK; ++i) p.Qhat[(u * DK + i) * DK + col] = X(i);
    } else {
#pragma unroll
      for (int i = 0; i < DK; ++i) p.S[(u * DK + i) * DV + col] = X(i);
    }
    if (tid == 0) {
      p.exp2[u] = exp2_acc;
      p.log_T[u] = static_cast<float>(logG);
    }
  } else {
#pragma unroll
    for (int i = 0; i < DK; ++i) p.S[(u * DK + i) * DV + col] = X(i);
    if (KIND == 1 && tid == 0)
      p.log_T[u] = static_cast<float>(static_cast<double>(it.len) *
                                      static_cast<double>(p.log_alpha[stream]));
    if (KIND == 3 && tid == 0) p.log_T[u] = 0.f;
    if (KIND == 4 && tid == 0) p.log_T[u] = static_cast<float>(logG);
    if (KIND == 2 && tid < DK) p.log_T[u * DK + tid] = static_cast<float>(logG);
  }
}

template <typename Tin, int D>
static cudaError_t launch_recur_t(const BuildParams& p, cudaStream_t st) {
  const dim3 grid(p.n_items);
  switch (p.kind) {
    case HYPIC_GDN:
      build_recurrence_kernel<Tin, D, D, 0><<<grid, 2 * D, 0, st>>>(p);
      break;
    case HYPIC_SCALAR_DECAY:
      build_recurrence_kernel<Tin, D, D, 1><<<grid, D, 0, st>>>(p);
      break;
    case HYPIC_DIAG_DECAY:
      build_recurrence_kernel<Tin, D, D, 2><<<grid, D, 0, st>>>(p);
      break;
    case HYPIC_TOKEN_DECAY:
      build_recurrence_kernel<Tin, D, D, 4><<<grid, D, 0, st>>>(p);
      break;
    case HYPIC_KDA:
      build_recurrence_kernel<Tin, D, D, 5><<<grid, 2 * D, 0, st>>>(p);
      break;
    default:
      build_recurrence_kernel<Tin, D, D, 3><<<grid, D, 0, st>>>(p);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_build_recurrence(const BuildParams& p, int in_dtype, cudaStream_t st) {
  if (in_dtype == HYPIC_F32)
    return p.dk == 64 ? launch_recur_t<float, 64>(p, st) : launch_recur_t<float, 128>(p, st);
  return p.dk == 64 ? launch_recur_t<__nv_bfloat16, 64>(p, st)
                    : launch_recur_t<__nv_bfloat16, 128>(p, st);
}

}  // namespace hypic
