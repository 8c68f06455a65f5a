// Compose cached pairs in request order, with the seam window of every
// position advanced first (youleyou.com HYPIC article: linear-layer paragraph
// for S <- T_C S + S(C|0); seam-window paragraph for the w seam tokens that
// are run under the full prefix and emit per-token outputs).
//
// One CTA per (request, stream) chain; thread m owns column m of the running
// state S (dk x dv, fp32 registers).  Per position j:
//   seam:    for each seam token t, by family (the same transitions as the build):
//              gated delta  u = k.x;  x <- alpha x + k (beta v_m - alpha beta u)
//              KDA          y = a o x;  u = k.y;  x <- y + k (beta v_m - beta u)
//              decay only   x <- a o x + k v_m  (a: per token, per stream or per
//                           key channel; 1 without decay)
//            then o_t[m] = q . x
//   compose: x <- c * Qhat_j x + S_j[:, m]   (gdn, c = e^logT 2^exp2; Qhat_j
//            staged in shared memory and read as broadcast rows)
//            x <- e^logT x + S_j[:, m]       (scalar / none)
//            x <- e^logT[i] x[i] + S_j[i, m] (diag)
#include <cuda_bf16.h>

#include "hypic_internal.h"

namespace hypic {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

// FAM: the seam tokens' family (hypic_kind)
template <int D, typename Tin, int FAM>
__global__ void __launch_bounds__(D) compose_kernel(ComposeParams p) {
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                 // [D][D] (gdn only)
  float* Ys = smem + D * D;         // [D][D] new state columns (gdn only)
  float* ks = Ys + D * D;           // [D]
  float* qs = ks + D;               // [D]
  float* as = qs + D;               // [D] per-channel decay of the token (GLA, KDA)
  constexpr bool kDelta = (FAM == HYPIC_GDN || FAM == HYPIC_KDA);
  constexpr bool kChan = (FAM == HYPIC_DIAG_DECAY || FAM == HYPIC_KDA);
  const int tid = threadIdx.x;
  const int chain = blockIdx.x;
  const int r = chain / p.n_streams;
  const int s = chain % p.n_streams;
  const int S = p.n_streams;

  float x[D];
  const int64_t st_base = (static_cast<int64_t>(r) * S + s) * D * D;
  if (p.state_in) {
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = p.state_in[st_base + i * D + tid];
  } else {
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = 0.f;
  }
  const Tin* qp = static_cast<const Tin*>(p.q);
  const Tin* kp = static_cast<const Tin*>(p.k);
  const Tin* vp = static_cast<const Tin*>(p.v);

  for (int j = 0; j < p.n_pos; ++j) {
    // ---- seam window of position j ----
    for (int t = 0; t < p.w; ++t) {
      const int64_t tok = ((static_cast<int64_t>(r) * p.n_pos + j) * p.w + t) * S + s;
      __syncthreads();
      ks[tid] = ld_f(kp, tok * D + tid);
      qs[tid] = ld_f(qp, tok * D + tid);
      if (kChan) as[tid] = expf(p.log_alpha[tok * D + tid]);
      __syncthreads();
      const float vm = ld_f(vp, tok * D + tid);
      // scalar decay of the token (1 for the per-channel and no-decay families)
      float al = 1.f;
      if (FAM == HYPIC_GDN || FAM == HYPIC_TOKEN_DECAY) al = expf(p.log_alpha[tok]);
      if (FAM == HYPIC_SCALAR_DECAY) al = expf(p.log_alpha[s]);
      if (kChan) {
#pragma unroll
        for (int i = 0; i < D; i += 4) {
          const float4 aa = *reinterpret_cast<const float4*>(&as[i]);
          x[i] *= aa.x;
          x[i + 1] *= aa.y;
          x[i + 2] *= aa.z;
          x[i + 3] *= aa.w;
        }
      }
      // write coefficient of k: beta (v_m - alpha k.x) for the delta rules, v_m otherwise
      float c = vm;
      if (kDelta) {
        const float be = p.beta[tok];
        float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
        for (int i = 0; i < D; i += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(&ks[i]);
          u0 = fmaf(kk.x, x[i], u0);
          u1 = fmaf(kk.y, x[i + 1], u1);
          u2 = fmaf(kk.z, x[i + 2], u2);
          u3 = fmaf(kk.w, x[i + 3], u3);
        }
        const float u = (u0 + u1) + (u2 + u3);
        c = be * vm - al * be * u;
      }
      float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
      for (int i = 0; i < D; i += 4) {
        const float4 kk = *reinterpret_cast<const float4*>(&ks[i]);
        const float4 qq = *reinterpret_cast<const float4*>(&qs[i]);
        x[i] = fmaf(al, x[i], kk.x * c);
        x[i + 1] = fmaf(al, x[i + 1], kk.y * c);
        x[i + 2] = fmaf(al, x[i + 2], kk.z * c);
        x[i + 3] = fmaf(al, x[i + 3], kk.w * c);
        o0 = fmaf(qq.x, x[i], o0);
        o1 = fmaf(qq.y, x[i + 1], o1);
        o2 = fmaf(qq.z, x[i + 2], o2);
        o3 = fmaf(qq.w, x[i + 3], o3);
      }
      store_o(p, tok * D + tid, (o0 + o1) + (o2 + o3));
    }
    if (p.kind < 0) continue;  // seam window only
    // ---- compose the cached pair of position j ----
    const int seg = p.order[static_cast<int64_t>(r) * p.n_pos + j];
    if (seg < 0 || seg >= p.n_seg) {
      if (tid == 0) report(p.ws, HYPIC_ERR_INDEX, 10);
      continue;
    }
    const int64_t u = static_cast<int64_t>(seg) * S + s;
    const float* __restrict__ Sj = p.Sc + u * D * D;
    if (p.kind == HYPIC_GDN) {
      const float c = expf(p.log_T[u] + static_cast<float>(p.exp2[u]) * 0.69314718055994531f);
      const float4* __restrict__ Qg = reinterpret_cast<const float4*>(p.Qhat + u * D * D);
      __syncthreads();
      for (int e = tid; e < D * D / 4; e += D) reinterpret_cast<float4*>(Qs)[e] = Qg[e];
      __syncthreads();
#pragma unroll 4
      for (int i = 0; i < D; ++i) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int kk = 0; kk < D; kk += 4) {
          const float4 qv = *reinterpret_cast<const float4*>(&Qs[i * D + kk]);
          a0 = fmaf(qv.x, x[kk], a0);
          a1 = fmaf(qv.y, x[kk + 1], a1);
          a2 = fmaf(qv.z, x[kk + 2], a2);
          a3 = fmaf(qv.w, x[kk + 3], a3);
        }
        Ys[i * D + tid] = fmaf(c, (a0 + a1) + (a2 + a3), Sj[i * D + tid]);
      }
#pragma unroll
      for (int i = 0; i < D; ++i) x[i] = Ys[i * D + tid];
    } else if (p.kind == HYPIC_DIAG_DECAY) {
#pragma unroll
      for (int i = 0; i < D; ++i) x[i] = fmaf(expf(p.log_T[u * D + i]), x[i], Sj[i * D + tid]);
    } else {
      const float c = expf(p.log_T[u]);
#pragma unroll
      for (int i = 0; i < D; ++i) x[i] = fmaf(c, x[i], Sj[i * D + tid]);
    }
  }
#pragma unroll
  for (int i = 0; i < D; ++i) p.state_out[st_base + i * D + tid] = x[i];
}

template <int D, typename Tin, int FAM>
static cudaError_t launch_compose_t(const ComposeParams& p, cudaStream_t st) {
  const size_t smem = (2 * static_cast<size_t>(D) * D + 3 * D) * sizeof(float);
  auto kern = compose_kernel<D, Tin, FAM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<p.n_req * p.n_streams, D, smem, st>>>(p);
  return cudaGetLastError();
}

template <int FAM>
static cudaError_t launch_compose_f(const ComposeParams& p, cudaStream_t st) {
  const bool f32 = (p.w > 0 && p.seam_dtype == HYPIC_F32);
  if (p.dk == 64)
    return f32 ? launch_compose_t<64, float, FAM>(p, st)
               : launch_compose_t<64, __nv_bfloat16, FAM>(p, st);
  return f32 ? launch_compose_t<128, float, FAM>(p, st)
             : launch_compose_t<128, __nv_bfloat16, FAM>(p, st);
}

cudaError_t launch_compose(const ComposeParams& p, cudaStream_t st) {
  switch (p.w > 0 ? p.seam_kind : HYPIC_GDN) {
    case HYPIC_SCALAR_DECAY: return launch_compose_f<HYPIC_SCALAR_DECAY>(p, st);
    case HYPIC_DIAG_DECAY: return launch_compose_f<HYPIC_DIAG_DECAY>(p, st);
    case HYPIC_NO_DECAY: return launch_compose_f<HYPIC_NO_DECAY>(p, st);
    case HYPIC_TOKEN_DECAY: return launch_compose_f<HYPIC_TOKEN_DECAY>(p, st);
    case HYPIC_KDA: return launch_compose_f<HYPIC_KDA>(p, st);
    default: return launch_compose_f<HYPIC_GDN>(p, st);
  }
}

}  // namespace hypic
