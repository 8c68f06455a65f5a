// Split build of long segments: the helper kernels.
//
// A segment's body is cut into pieces that are built as ordinary pairs in
// parallel; by the composition law of the pairs (youleyou.com HYPIC article,
// linear-layer paragraph: T(C2 C1) = T(C2) T(C1), S(C2 C1) = T(C2) S(C1) +
// S(C2)) the segment's pair is the ordered composition of its pieces' pairs.
// The host side runs that composition with the compose kernels (S from zero;
// for the gated-delta Qhat, the product of the pieces' Qhat from I with the
// decays and S set to zero); the kernels here prepare the identity pair and
// the start states and finish the factored T: log T summed over the pieces,
// the power-of-two exponents summed, Qhat renormalised by an exact power of two.
#include "hypic_internal.h"

namespace hypic {

// Identity pair (Qhat = I, exp2 = 0, log T = 0, S = 0) at unit index `unit0`
// .. unit0 + n_streams - 1, and (when `eye` is not null) identity matrices for
// n_units start states.  One CTA per matrix, 128 threads (dk = dv <= 128).
__global__ void split_fill_kernel(float* Qhat, int32_t* exp2, float* log_T, int log_T_width,
                                  float* S, int64_t unit0, int n_streams, int d, float* eye,
                                  int64_t n_eye) {
  const int64_t m = blockIdx.x;
  const int t = threadIdx.x;
  if (m < n_streams) {
    const int64_t u = unit0 + m;
    for (int e = t; e < d * d; e += blockDim.x) {
      if (Qhat) Qhat[u * d * d + e] = (e / d == e % d) ? 1.f : 0.f;
      S[u * d * d + e] = 0.f;
    }
    if (t < log_T_width) log_T[u * log_T_width + t] = 0.f;
    if (t == 0 && exp2) exp2[u] = 0;
  } else if (eye && m - n_streams < n_eye) {
    const int64_t u = m - n_streams;
    for (int e = t; e < d * d; e += blockDim.x) eye[u * d * d + e] = (e / d == e % d) ? 1.f : 0.f;
  }
}

// Per output unit (segment i, stream s): log T (scalar or per channel) and the
// exponent summed over the segment's pieces in `order` (padding = the identity
// unit, which adds nothing); Qhat (already the product of the pieces' Qhat)
// renormalised so that max |Qhat| is in [1, 2).  Also folds the compose call's
// device status into the build's status word.  One CTA per unit, 128 threads.
__global__ void split_finish_kernel(const int32_t* order, int n_pos, int n_streams, int d,
                                    const float* sub_log_T, const int32_t* sub_exp2,
                                    int log_T_width, float* log_T, int32_t* exp2, float* Qhat,
                                    WsHeader* ws, const WsHeader* ws_c1, const WsHeader* ws_c2) {
  __shared__ float red[32];
  const int64_t u = blockIdx.x;
  const int64_t seg = u / n_streams;
  const int s = static_cast<int>(u % n_streams);
  const int t = threadIdx.x;
  if (u == 0 && t == 0) {
    if (ws_c1->status) report(ws, ws_c1->status, ws_c1->where);
    if (ws_c2 && ws_c2->status) report(ws, ws_c2->status, ws_c2->where);
  }
  if (t < log_T_width) {
    double acc = 0.0;
    for (int j = 0; j < n_pos; ++j) {
      const int64_t su = static_cast<int64_t>(order[seg * n_pos + j]) * n_streams + s;
      acc += static_cast<double>(sub_log_T[su * log_T_width + t]);
    }
    log_T[u * log_T_width + t] = static_cast<float>(acc);
  }
  if (!Qhat) return;
  int e_sum = 0;
  for (int j = 0; j < n_pos; ++j)
    e_sum += sub_exp2[static_cast<int64_t>(order[seg * n_pos + j]) * n_streams + s];
  float m = 0.f;
  float* q = Qhat + u * d * d;
  for (int e = t; e < d * d; e += blockDim.x) m = fmaxf(m, fabsf(q[e]));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  float mm = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) mm = fmaxf(mm, red[w]);
  int sh = 0;
  if (mm > 0.f) {
    int e2;
    frexpf(mm, &e2);   // mm = f 2^e2, f in [0.5, 1)
    sh = 1 - e2;       // mm 2^sh in [1, 2)
  }
  if (sh != 0)
    for (int e = t; e < d * d; e += blockDim.x) q[e] = ldexpf(q[e], sh);
  if (t == 0) exp2[u] = e_sum - sh;
}

cudaError_t launch_split_fill(float* Qhat, int32_t* exp2, float* log_T, int log_T_width, float* S,
                              int64_t unit0, int n_streams, int d, float* eye, int64_t n_eye,
                              cudaStream_t st) {
  const int64_t blocks = n_streams + (eye ? n_eye : 0);
  if (blocks == 0) return cudaSuccess;
  split_fill_kernel<<<static_cast<unsigned>(blocks), 128, 0, st>>>(
      Qhat, exp2, log_T, log_T_width, S, unit0, n_streams, d, eye, n_eye);
  return cudaGetLastError();
}

cudaError_t launch_split_finish(const int32_t* order, int n_pos, int64_t n_units, int n_streams,
                                int d, const float* sub_log_T, const int32_t* sub_exp2,
                                int log_T_width, float* log_T, int32_t* exp2, float* Qhat,
                                WsHeader* ws, const WsHeader* ws_c1, const WsHeader* ws_c2,
                                cudaStream_t st) {
  if (n_units == 0) return cudaSuccess;
  split_finish_kernel<<<static_cast<unsigned>(n_units), 128, 0, st>>>(
      order, n_pos, n_streams, d, sub_log_T, sub_exp2, log_T_width, log_T, exp2, Qhat, ws, ws_c1,
      ws_c2);
  return cudaGetLastError();
}

}  // namespace hypic
