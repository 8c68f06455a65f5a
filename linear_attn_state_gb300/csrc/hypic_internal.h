// Internal declarations shared by the host dispatcher and the kernels of
// libhypic.so.  Nothing here is part of the public ABI (include/hypic.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/hypic.h"

namespace hypic {

// One build work item: the body of one (segment, stream) unit.
struct WorkItem {
  int64_t tok_start;  // first body token (packed index)
  int32_t len;        // body length in tokens (may be 0)
  int32_t unit;       // seg * n_streams + stream
};
static_assert(sizeof(WorkItem) == 16, "WorkItem layout");

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
  int32_t status;     // first device-detected error (hypic_status), 0 = none
  uint32_t queue;     // persistent-kernel work counter
  int32_t where;      // diagnostic: site id of the first error
  int32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "WsHeader layout");

constexpr size_t kWsHeaderBytes = 256;

// Compose workspace, after the header: seam chunk records, then (when the
// cached pairs are reused enough) the operand copy of every pair's Qhat.
// Seam windows on the tensor-core compose are cut into chunks of up to
// kSeamChunk tokens; the state-independent part of each chunk (per stream) is
// precomputed into one record of kSeamRecordBytes.
constexpr int kSeamChunk = 8;
constexpr size_t kSeamRecordBytes = 16896;
// Operand copy of a 128 x 128 Qhat: fp16 hi and lo planes in the tensor-core
// B layout (64 KB), and one power-of-two exponent per pair.
constexpr size_t kQopBytes = 65536;

struct ComposeWsLayout {
  size_t rec = 0, qop = 0, qexp = 0, bytes = 0;   // byte offsets (0: absent), total
};
inline size_t ws_round(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
// The layout for a compose over n_req x n_pos positions of a cache with n_seg
// pairs of n_streams streams.  The tensor-core path (gated-delta form, dk = dv =
// 128) uses records for a seam window and, when the positions reuse each pair
// twice or more on average, the operand copy.
inline ComposeWsLayout compose_ws_layout(int64_t n_seg, int64_t n_streams, int dk, int dv,
                                         bool matrix_form, int64_t n_req, int64_t n_pos, int64_t w) {
  ComposeWsLayout L;
  size_t o = kWsHeaderBytes;
  const bool tc = matrix_form && dk == 128 && dv == 128 && n_seg > 0 && n_streams > 0;
  if (tc && w > 0 && n_req > 0 && n_pos > 0) {
    const int64_t nch = (w + kSeamChunk - 1) / kSeamChunk;
    L.rec = o;
    o += ws_round(static_cast<size_t>(n_req * n_pos * nch * n_streams) * kSeamRecordBytes);
  }
  if (tc && n_req > 0 && n_req * n_pos >= 2 * n_seg) {
    const size_t units = static_cast<size_t>(n_seg * n_streams);
    L.qop = o;
    o += ws_round(units * kQopBytes);
    L.qexp = o;
    o += ws_round(units * 4);
  }
  L.bytes = o;
  return L;
}

// Record a device error once (first error wins).
__device__ __forceinline__ void report(WsHeader* ws, int code, int where) {
  if (atomicCAS(&ws->status, 0, code) == 0) ws->where = where;
}

// Device view of build inputs (k/v typed by the kernel template).
struct BuildParams {
  const WorkItem* items;
  int32_t n_items;
  int32_t n_streams;
  int32_t dk, dv;
  int32_t kind;
  int64_t n_tok;
  const void* k;
  const void* v;
  const float* beta;
  const float* log_alpha;
  float* Qhat;
  int32_t* exp2;
  float* log_T;
  float* S;
  WsHeader* ws;
  uint32_t spin_limit;
  int32_t redo_only;   // recurrence: build only the units whose exp2 holds kKdaRedo
};

// exp2 of a KDA unit that the tensor-core build leaves to the token recurrence
// (a chunk's decay span beyond its single-reference bound); never a real exponent.
constexpr int32_t kKdaRedo = INT32_MIN;

struct ComposeParams {
  int32_t n_req, n_pos, n_seg, n_streams, dk, dv, kind;
  const int32_t* order;
  const float* Qhat;
  const int32_t* exp2;
  const float* log_T;
  const float* Sc;         // cached S
  const float* state_in;   // may be null
  float* state_out;
  // seam (w == 0 when absent)
  int32_t w;
  int32_t seam_dtype;
  int32_t seam_kind;       // hypic_kind of the seam tokens' transitions
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* log_alpha;
  void* out_o;
  int32_t o_bf16;          // out_o holds bf16 (else fp32)
  uint8_t* seam_rec;       // tensor-core compose: the seam chunk records (workspace)
  uint8_t* qop;            // tensor-core compose: operand copies of Qhat (workspace) or null
  int32_t* qop_exp;        //   and their exponents
  WsHeader* ws;
  uint32_t spin_limit;
};

// Seam output o_t element i: fp32, or bf16 rounded to nearest even.
__device__ __forceinline__ void store_o(const ComposeParams& p, int64_t i, float v) {
  if (p.o_bf16)
    static_cast<__nv_bfloat16*>(p.out_o)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p.out_o)[i] = v;
}

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_build_recurrence(const BuildParams& p, int in_dtype, cudaStream_t st);
cudaError_t launch_build_decay(const BuildParams& p, int n_ctas, cudaStream_t st);
cudaError_t launch_build_gdn_tc(const BuildParams& p, int n_ctas, cudaStream_t st);
cudaError_t launch_build_kda_tc(const BuildParams& p, int n_ctas, cudaStream_t st);
// 3-D tensor map over packed tokens [n_tok][n_streams][d] bf16: boxes of 64 tokens x
// 1 stream x 64 channels (128 bytes), 128-byte swizzle (the K-major operand layout).
bool make_token_map(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams, int d);
// The same over per-channel gates [n_tok][n_streams][d] fp32: boxes of 64 tokens x
// 1 stream x 32 channels (128 bytes), 128-byte swizzle: [64 t][32 i] per box with
// the 16-byte chunks of row t permuted by XOR with t mod 8.
bool make_gate_map(CUtensorMap* m, const float* base, int64_t n_tok, int n_streams, int d);
cudaError_t launch_compose(const ComposeParams& p, cudaStream_t st);
bool compose_tc_supported(const ComposeParams& p);
cudaError_t launch_compose_tc(const ComposeParams& p, cudaStream_t st);

cudaError_t launch_split_fill(float* Qhat, int32_t* exp2, float* log_T, int log_T_width, float* S,
                              int64_t unit0, int n_streams, int d, float* eye, int64_t n_eye,
                              cudaStream_t st);
cudaError_t launch_split_finish(const int32_t* order, int n_pos, int64_t n_units, int n_streams,
                                int d, const float* sub_log_T, const int32_t* sub_exp2,
                                int log_T_width, float* log_T, int32_t* exp2, float* Qhat,
                                WsHeader* ws, const WsHeader* ws_c1, const WsHeader* ws_c2,
                                cudaStream_t st);

uint32_t current_spin_limit();
// The host checks of hypic_segment_build (arguments, cache, device arch), in
// its order; HYPIC_OK when a build with these arguments may launch.
hypic_status check_build_call(const hypic_build_args* a, const hypic_cache* out);
int device_sm_count();

}  // namespace hypic
