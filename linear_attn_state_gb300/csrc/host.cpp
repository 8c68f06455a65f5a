// Host side of libhypic.so: argument validation, LPT scheduling, workspace
// sizing and kernel dispatch behind the C ABI of include/hypic.h.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "hypic_internal.h"

namespace hypic {

namespace {
constexpr uint32_t kDefaultSpinLimit = 1u << 21;  // suspending polls of <= ~2 us each
std::atomic<uint32_t> g_spin_limit{kDefaultSpinLimit};
std::atomic<int32_t> g_build_order{HYPIC_ORDER_LPT};

struct DevInfo {
  int ok = -1;  // -1 unknown, 0 wrong arch, 1 sm_103
  int sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

// Checks that the current device is sm_103 (GB300) and caches its SM count.
hypic_status check_arch(int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (dev < 0 || dev >= 64) return HYPIC_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return HYPIC_ERR_CUDA;
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
    d.sms = sms;
  }
  if (sms_out) *sms_out = d.sms;
  return d.ok == 1 ? HYPIC_OK : HYPIC_ERR_ARCH;
}

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
// Arrays the kernels read with 16-byte vector loads or tensor-memory copies
// (TMA) start on a 16-byte boundary; NULL passes (checked elsewhere).
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool offsets_ok(const int64_t* off, int32_t n_seg, int64_t n_tok) {
  if (off[0] != 0) return false;
  for (int32_t i = 0; i < n_seg; ++i)
    if (off[i + 1] < off[i]) return false;
  return off[n_seg] == n_tok;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

uint32_t current_spin_limit() { return g_spin_limit.load(); }

int device_sm_count() {
  int sms = 0;
  check_arch(&sms);
  return sms > 0 ? sms : 1;
}

cudaError_t launch_build_prepare(const int64_t* d_offsets, int32_t n_seg, int32_t seam_w,
                                 int32_t n_streams, int64_t n_tok, int64_t tok_base,
                                 int32_t seg_off, bool index_order, WorkItem* items, WsHeader* ws,
                                 cudaStream_t st);

}  // namespace hypic

using namespace hypic;

extern "C" {

int32_t hypic_version(void) { return 100; }

const char* hypic_status_str(hypic_status s) {
  switch (s) {
    case HYPIC_OK: return "HYPIC_OK";
    case HYPIC_ERR_NULL: return "HYPIC_ERR_NULL";
    case HYPIC_ERR_SHAPE: return "HYPIC_ERR_SHAPE";
    case HYPIC_ERR_OFFSETS: return "HYPIC_ERR_OFFSETS";
    case HYPIC_ERR_INDEX: return "HYPIC_ERR_INDEX";
    case HYPIC_ERR_DTYPE: return "HYPIC_ERR_DTYPE";
    case HYPIC_ERR_WORKSPACE: return "HYPIC_ERR_WORKSPACE";
    case HYPIC_ERR_ARCH: return "HYPIC_ERR_ARCH";
    case HYPIC_ERR_CUDA: return "HYPIC_ERR_CUDA";
    case HYPIC_ERR_DEVICE_TIMEOUT: return "HYPIC_ERR_DEVICE_TIMEOUT";
  }
  return "HYPIC_ERR_UNKNOWN";
}

uint32_t hypic_set_spin_limit(uint32_t limit) {
  // kernels receive the number of polls; HYPIC_SPIN_EXPIRE_NOW is zero polls
  const uint32_t polls =
      limit == 0 ? kDefaultSpinLimit : (limit == HYPIC_SPIN_EXPIRE_NOW ? 0u : limit);
  const uint32_t prev = g_spin_limit.exchange(polls);
  return prev == 0 ? HYPIC_SPIN_EXPIRE_NOW : prev;
}

int32_t hypic_set_build_order(int32_t order) {
  if (order != HYPIC_ORDER_LPT && order != HYPIC_ORDER_INDEX) return -1;
  return g_build_order.exchange(order);
}

hypic_status hypic_offsets_from_lengths(const int64_t* h_len, int32_t n, int64_t* h_offsets) {
  if (n < 0) return HYPIC_ERR_SHAPE;
  if (!h_offsets || (n > 0 && !h_len)) return HYPIC_ERR_NULL;
  for (int32_t i = 0; i < n; ++i)
    if (h_len[i] < 0) return HYPIC_ERR_SHAPE;
  h_offsets[0] = 0;
  for (int32_t i = 0; i < n; ++i) h_offsets[i + 1] = h_offsets[i] + h_len[i];
  return HYPIC_OK;
}

hypic_status hypic_lpt_schedule(const int64_t* h_offsets, int32_t n_seg, int32_t seam_w,
                                int32_t n_streams, int32_t n_workers, int32_t* h_order,
                                int32_t* h_worker) {
  if (!h_offsets || (!h_order && n_seg > 0)) return HYPIC_ERR_NULL;
  if (n_seg < 0 || n_streams < 1 || n_workers < 1 || seam_w < 0) return HYPIC_ERR_SHAPE;
  if (static_cast<int64_t>(n_seg) * n_streams > INT32_MAX) return HYPIC_ERR_SHAPE;
  if (!offsets_ok(h_offsets, n_seg, h_offsets[n_seg])) return HYPIC_ERR_OFFSETS;
  // Body costs; segment order by (-cost, seg); streams ascending inside a
  // segment give the (-cost, seg, stream) item order.
  std::vector<int64_t> cost(n_seg);
  std::vector<int32_t> segs(n_seg);
  for (int32_t i = 0; i < n_seg; ++i) {
    const int64_t L = h_offsets[i + 1] - h_offsets[i];
    cost[i] = L - std::min<int64_t>(seam_w, L);
    segs[i] = i;
  }
  std::stable_sort(segs.begin(), segs.end(),
                   [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });
  using Slot = std::pair<int64_t, int32_t>;  // (load, worker id)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  if (h_worker)
    for (int32_t w = 0; w < n_workers; ++w) heap.push({0, w});
  int64_t pos = 0;
  for (int32_t r = 0; r < n_seg; ++r) {
    const int32_t seg = segs[r];
    for (int32_t s = 0; s < n_streams; ++s) {
      const int32_t item = seg * n_streams + s;
      h_order[pos++] = item;
      if (h_worker) {
        Slot top = heap.top();
        heap.pop();
        h_worker[item] = top.second;
        heap.push({top.first + cost[seg], top.second});
      }
    }
  }
  return HYPIC_OK;
}

size_t hypic_build_workspace_bytes(const hypic_build_args* a) {
  if (!a || a->n_seg < 0 || a->n_streams < 1) return 0;
  const size_t n_items = static_cast<size_t>(a->n_seg) * static_cast<size_t>(a->n_streams);
  return kWsHeaderBytes + round_up(n_items * sizeof(WorkItem), 256);
}

size_t hypic_compose_workspace_bytes(const hypic_cache* cache, int32_t n_req, int32_t n_pos,
                                     int32_t seam_w) {
  if (!cache) return 0;
  return compose_ws_layout(cache->n_seg, cache->n_streams, cache->dk, cache->dv,
                           cache->kind == HYPIC_GDN || cache->kind == HYPIC_KDA, n_req, n_pos,
                           seam_w)
      .bytes;
}

hypic_status hypic_read_device_status(const void* d_ws, void* stream, int32_t* h_status) {
  if (!d_ws || !h_status) return HYPIC_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return HYPIC_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, d_ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return HYPIC_ERR_CUDA;
  *h_status = v;
  return HYPIC_OK;
}

namespace hypic {
namespace {

// Families by what they read and cache: a delta rule reads beta; a "factored"
// cache holds T = exp(log_T) 2^exp2 Qhat (the matrix families); the per-token
// gate is one value (GDN, TOKEN) or dk values (DIAG, KDA) per token and stream.
bool has_beta(int kind) { return kind == HYPIC_GDN || kind == HYPIC_KDA; }
bool factored(int kind) { return kind == HYPIC_GDN || kind == HYPIC_KDA; }
size_t gate_floats(int kind, int dk) {
  if (kind == HYPIC_GDN || kind == HYPIC_TOKEN_DECAY) return 1;
  if (kind == HYPIC_DIAG_DECAY || kind == HYPIC_KDA) return static_cast<size_t>(dk);
  return 0;
}
int log_T_width(int kind, int dk) { return kind == HYPIC_DIAG_DECAY ? dk : 1; }

// Everything a build checks on the host, for args whose cache covers them.
hypic_status check_build_args(const hypic_build_args* a) {
  if (!a) return HYPIC_ERR_NULL;
  if (a->n_seg < 0 || a->n_streams < 1 || a->seam_w < 0 || a->n_tok < 0) return HYPIC_ERR_SHAPE;
  // token coordinates are 32-bit on the device (tensor-map coordinates, work-item lengths)
  if (a->n_tok > INT32_MAX) return HYPIC_ERR_SHAPE;
  if (!(a->dk == a->dv && (a->dk == 64 || a->dk == 128))) return HYPIC_ERR_SHAPE;
  if (a->kind < HYPIC_GDN || a->kind > HYPIC_KDA) return HYPIC_ERR_DTYPE;
  if (a->in_dtype != HYPIC_BF16 && a->in_dtype != HYPIC_F32) return HYPIC_ERR_DTYPE;
  if (!a->h_offsets || !a->d_offsets) return HYPIC_ERR_NULL;
  if (a->n_tok > 0 && (!a->k || !a->v)) return HYPIC_ERR_NULL;
  if (has_beta(a->kind) && a->n_tok > 0 && !a->beta) return HYPIC_ERR_NULL;
  if (gate_floats(a->kind, a->dk) > 0 && a->n_tok > 0 && !a->log_alpha) return HYPIC_ERR_NULL;
  if (a->kind == HYPIC_SCALAR_DECAY && !a->log_alpha) return HYPIC_ERR_NULL;
  if (static_cast<int64_t>(a->n_seg) * a->n_streams > INT32_MAX) return HYPIC_ERR_SHAPE;
  if (!offsets_ok(a->h_offsets, a->n_seg, a->n_tok)) return HYPIC_ERR_OFFSETS;
  return HYPIC_OK;
}

hypic_status check_cache(const hypic_build_args* a, const hypic_cache* out) {
  if (!out) return HYPIC_ERR_NULL;
  if (out->n_seg != a->n_seg || out->n_streams != a->n_streams || out->dk != a->dk ||
      out->dv != a->dv || out->kind != a->kind)
    return HYPIC_ERR_SHAPE;
  const int64_t n_items64 = static_cast<int64_t>(a->n_seg) * a->n_streams;
  if (n_items64 > 0 && (!out->S || !out->log_T)) return HYPIC_ERR_NULL;
  if (n_items64 > 0 && factored(a->kind) && (!out->Qhat || !out->exp2)) return HYPIC_ERR_NULL;
  if (!aligned16(out->S) || !aligned16(out->Qhat)) return HYPIC_ERR_SHAPE;
  return HYPIC_OK;
}

// Device-resident inputs of a build (not the host-input entry, whose inputs are
// staged into aligned device buffers): keys, values and per-channel gates.
hypic_status check_device_inputs(const hypic_build_args* a) {
  if (!aligned16(a->k) || !aligned16(a->v)) return HYPIC_ERR_SHAPE;
  if (gate_floats(a->kind, a->dk) > 1 && !aligned16(a->log_alpha)) return HYPIC_ERR_SHAPE;
  return HYPIC_OK;
}

// The launches of one build over the n_seg segments of `a` (validated), whose
// offsets are read on the device as a->d_offsets[i] - tok_base and whose units
// are written at segment index seg_off + i of `out`.
hypic_status launch_build(const hypic_build_args* a, const hypic_cache* out, void* d_ws,
                          cudaStream_t st, int64_t tok_base, int32_t seg_off, int sms) {
  WsHeader* ws = static_cast<WsHeader*>(d_ws);
  WorkItem* items = reinterpret_cast<WorkItem*>(static_cast<char*>(d_ws) + kWsHeaderBytes);
  if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return HYPIC_ERR_CUDA;
  const int32_t n_items = a->n_seg * a->n_streams;
  if (n_items == 0) return HYPIC_OK;
  if (launch_build_prepare(a->d_offsets, a->n_seg, a->seam_w, a->n_streams, a->n_tok, tok_base,
                           seg_off, g_build_order.load() == HYPIC_ORDER_INDEX, items, ws,
                           st) != cudaSuccess)
    return HYPIC_ERR_CUDA;

  BuildParams p{};
  p.items = items;
  p.n_items = n_items;
  p.n_streams = a->n_streams;
  p.dk = a->dk;
  p.dv = a->dv;
  p.kind = a->kind;
  p.n_tok = a->n_tok;
  p.k = a->k;
  p.v = a->v;
  p.beta = a->beta;
  p.log_alpha = a->log_alpha;
  p.Qhat = out->Qhat;
  p.exp2 = out->exp2;
  p.log_T = out->log_T;
  p.S = out->S;
  p.ws = ws;
  p.spin_limit = current_spin_limit();

  cudaError_t e;
  if (a->kind == HYPIC_GDN && a->in_dtype == HYPIC_BF16)
    e = launch_build_gdn_tc(p, sms, st);
  else if (a->kind == HYPIC_KDA && a->in_dtype == HYPIC_BF16)
    e = launch_build_kda_tc(p, sms, st);
  else if (a->kind == HYPIC_GDN || a->kind == HYPIC_KDA || a->in_dtype == HYPIC_F32)
    e = launch_build_recurrence(p, a->in_dtype, st);
  else
    e = launch_build_decay(p, sms, st);
  return e == cudaSuccess ? HYPIC_OK : HYPIC_ERR_CUDA;
}

// Segment groups of a host-input build: consecutive segments while the group's
// token count stays within max_tokens (a longer segment forms its own group).
std::vector<int32_t> segment_groups(const int64_t* off, int32_t n_seg, int64_t max_tokens) {
  std::vector<int32_t> starts;
  int32_t i = 0;
  while (i < n_seg) {
    starts.push_back(i);
    int32_t j = i + 1;
    while (j < n_seg && off[j + 1] - off[i] <= max_tokens) ++j;
    i = j;
  }
  starts.push_back(n_seg);
  return starts;
}

// Bytes of one staging half for `tokens` tokens, and the offsets of k, v, beta
// and log_alpha in it (256-byte aligned).
struct StageLayout {
  size_t k, v, beta, log_alpha, bytes;
};
StageLayout stage_layout(const hypic_build_args* a, int64_t tokens) {
  const size_t es = (a->in_dtype == HYPIC_F32) ? 4 : 2;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  StageLayout L{};
  const size_t T = static_cast<size_t>(tokens), S = static_cast<size_t>(a->n_streams);
  L.k = 0;
  L.v = up(T * S * a->dk * es);
  L.beta = L.v + up(T * S * a->dv * es);
  L.log_alpha = L.beta + (has_beta(a->kind) ? up(T * S * 4) : 0);
  size_t g = T * S * gate_floats(a->kind, a->dk) * 4;
  if (a->kind == HYPIC_SCALAR_DECAY) g = S * 4;
  L.bytes = L.log_alpha + up(g);
  return L;
}

// Pieces of a split build: every segment's seam window (when w > 0) is a piece
// of its own that no segment uses; its body is cut into pieces of at most
// piece_tokens tokens.  Pieces cover [0, n_tok) in order (their offsets are a
// valid offsets array); order[i][j] is the j-th body piece of segment i, padded
// with the identity unit n_pieces.
struct SplitPlan {
  std::vector<int64_t> off;      // n_pieces + 1
  std::vector<int32_t> order;    // n_seg * n_pos
  int32_t n_pieces = 0, n_pos = 1;
};
SplitPlan split_plan(const hypic_build_args* a, int64_t piece_tokens) {
  SplitPlan sp;
  sp.off.push_back(0);
  std::vector<std::vector<int32_t>> body(a->n_seg);
  for (int32_t i = 0; i < a->n_seg; ++i) {
    const int64_t b0 = a->h_offsets[i], e = a->h_offsets[i + 1], L = e - b0;
    const int64_t w = std::min<int64_t>(a->seam_w, L);
    if (w > 0) sp.off.push_back(b0 + w);
    for (int64_t pos = b0 + w; pos < e; pos += piece_tokens) {
      body[i].push_back(static_cast<int32_t>(sp.off.size() - 1));
      sp.off.push_back(std::min(pos + piece_tokens, e));
    }
    sp.n_pos = std::max<int32_t>(sp.n_pos, static_cast<int32_t>(body[i].size()));
  }
  sp.n_pieces = static_cast<int32_t>(sp.off.size() - 1);
  sp.order.assign(static_cast<size_t>(a->n_seg) * sp.n_pos, sp.n_pieces);
  for (int32_t i = 0; i < a->n_seg; ++i)
    for (size_t j = 0; j < body[i].size(); ++j) sp.order[static_cast<size_t>(i) * sp.n_pos + j] = body[i][j];
  return sp;
}

// Scratch of a split build, 256-byte aligned pieces: the build workspace first
// (its status word is the call's), the pieces' cache (+ the identity unit),
// the compose views' zero S / log T / exponents, the identity start states, the
// order, the pieces' device offsets, and two compose workspaces.
struct SplitLayout {
  size_t ws_b, c_q, c_e, c_l, c_s, z_s, z_l, z_e, eye, order, off, ws_c1, ws_c2, bytes;
};
SplitLayout split_layout(const hypic_build_args* a, const SplitPlan& sp) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t S = a->n_streams, d = a->dk, U = static_cast<size_t>(sp.n_pieces + 1) * S;
  const bool gdn = factored(a->kind);
  const size_t lw = static_cast<size_t>(log_T_width(a->kind, a->dk));
  hypic_build_args g = *a;
  g.n_seg = sp.n_pieces;
  SplitLayout L{};
  size_t o = 0;
  L.ws_b = o; o += up(hypic_build_workspace_bytes(&g));
  L.c_q = o; o += gdn ? up(U * d * d * 4) : 0;
  L.c_e = o; o += gdn ? up(U * 4) : 0;
  L.c_l = o; o += up(U * lw * 4);
  L.c_s = o; o += up(U * d * d * 4);
  L.z_s = o; o += gdn ? up(U * d * d * 4) : 0;
  L.z_l = o; o += gdn ? up(U * 4) : 0;
  L.z_e = o; o += gdn ? up(U * 4) : 0;
  L.eye = o; o += gdn ? up(static_cast<size_t>(a->n_seg) * S * d * d * 4) : 0;
  L.order = o; o += up(sp.order.size() * 4);
  L.off = o; o += up(sp.off.size() * 8);
  const size_t wc = compose_ws_layout(sp.n_pieces + 1, a->n_streams, a->dk, a->dv, gdn, a->n_seg,
                                      sp.n_pos, 0).bytes;
  L.ws_c1 = o; o += up(wc);
  L.ws_c2 = o; o += up(wc);
  L.bytes = o;
  return L;
}

}  // namespace
}  // namespace hypic

extern "C++" {
namespace hypic {
hypic_status check_build_call(const hypic_build_args* a, const hypic_cache* out) {
  hypic_status s = check_build_args(a);
  if (s != HYPIC_OK) return s;
  if ((s = check_cache(a, out)) != HYPIC_OK) return s;
  if ((s = check_device_inputs(a)) != HYPIC_OK) return s;
  return check_arch(nullptr);
}
}  // namespace hypic
}

hypic_status hypic_segment_build(const hypic_build_args* a, const hypic_cache* out, void* d_ws,
                                 size_t ws_bytes, void* stream) {
  hypic_status s = check_build_args(a);
  if (s != HYPIC_OK) return s;
  if ((s = check_cache(a, out)) != HYPIC_OK) return s;
  if ((s = check_device_inputs(a)) != HYPIC_OK) return s;
  if (!d_ws || !aligned256(d_ws) || ws_bytes < hypic_build_workspace_bytes(a))
    return HYPIC_ERR_WORKSPACE;
  int sms = 0;
  if ((s = check_arch(&sms)) != HYPIC_OK) return s;
  return launch_build(a, out, d_ws, static_cast<cudaStream_t>(stream), 0, 0, sms);
}

size_t hypic_build_host_stage_bytes(const hypic_build_args* a, int64_t max_group_tokens) {
  if (check_build_args(a) != HYPIC_OK || max_group_tokens < 1) return 0;
  const auto starts = segment_groups(a->h_offsets, a->n_seg, max_group_tokens);
  int64_t most = 0;
  for (size_t gi = 0; gi + 1 < starts.size(); ++gi)
    most = std::max(most, a->h_offsets[starts[gi + 1]] - a->h_offsets[starts[gi]]);
  return 2 * stage_layout(a, std::max<int64_t>(most, 1)).bytes;
}

hypic_status hypic_segment_build_host(const hypic_build_args* a, const hypic_cache* out,
                                      int64_t max_group_tokens, void* d_stage, size_t stage_bytes,
                                      void* d_ws, size_t ws_bytes, void* stream,
                                      void* copy_stream) {
  hypic_status s = check_build_args(a);
  if (s != HYPIC_OK) return s;
  if ((s = check_cache(a, out)) != HYPIC_OK) return s;
  if (max_group_tokens < 1) return HYPIC_ERR_SHAPE;
  if (!d_ws || !aligned256(d_ws) || ws_bytes < hypic_build_workspace_bytes(a))
    return HYPIC_ERR_WORKSPACE;
  const size_t need = hypic_build_host_stage_bytes(a, max_group_tokens);
  if (!d_stage || !aligned256(d_stage) || stage_bytes < need) return HYPIC_ERR_WORKSPACE;
  int sms = 0;
  if ((s = check_arch(&sms)) != HYPIC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  const auto starts = segment_groups(a->h_offsets, a->n_seg, max_group_tokens);
  const size_t half = need / 2;
  const size_t es = (a->in_dtype == HYPIC_F32) ? 4 : 2;
  const size_t S = static_cast<size_t>(a->n_streams);

  // events: a stage half copied / free again
  cudaEvent_t copied[2], freed[2];
  for (int h = 0; h < 2; ++h) {
    if (cudaEventCreateWithFlags(&copied[h], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&freed[h], cudaEventDisableTiming) != cudaSuccess)
      return HYPIC_ERR_CUDA;
  }
  // copies of this call start after the work already queued on `stream`
  hypic_status rc = HYPIC_OK;
  if (cudaEventRecord(freed[0], st) != cudaSuccess || cudaEventRecord(freed[1], st) != cudaSuccess)
    rc = HYPIC_ERR_CUDA;
  std::vector<int64_t> rel;   // the group's offsets rebased to its first token
  for (size_t gi = 0; rc == HYPIC_OK && gi + 1 < starts.size(); ++gi) {
    const int32_t s0 = starts[gi], s1 = starts[gi + 1];
    const int64_t t0 = a->h_offsets[s0], t1 = a->h_offsets[s1], T = t1 - t0;
    const int h = static_cast<int>(gi & 1);
    char* base = static_cast<char*>(d_stage) + h * half;
    const StageLayout L = stage_layout(a, std::max<int64_t>(T, 1));
    auto copy = [&](size_t dst_off, const void* src, size_t row_bytes) {
      if (T == 0) return cudaSuccess;
      return cudaMemcpyAsync(base + dst_off,
                             static_cast<const char*>(src) + static_cast<size_t>(t0) * row_bytes,
                             static_cast<size_t>(T) * row_bytes, cudaMemcpyHostToDevice, cs);
    };
    cudaError_t e = cudaStreamWaitEvent(cs, freed[h], 0);
    if (e == cudaSuccess) e = copy(L.k, a->k, S * a->dk * es);
    if (e == cudaSuccess) e = copy(L.v, a->v, S * a->dv * es);
    if (e == cudaSuccess && has_beta(a->kind)) e = copy(L.beta, a->beta, S * 4);
    if (e == cudaSuccess && gate_floats(a->kind, a->dk) > 0)
      e = copy(L.log_alpha, a->log_alpha, S * gate_floats(a->kind, a->dk) * 4);
    if (e == cudaSuccess && a->kind == HYPIC_SCALAR_DECAY)
      e = cudaMemcpyAsync(base + L.log_alpha, a->log_alpha, S * 4, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(copied[h], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, copied[h], 0);
    if (e != cudaSuccess) { rc = HYPIC_ERR_CUDA; break; }

    hypic_build_args g = *a;
    rel.assign(a->h_offsets + s0, a->h_offsets + s1 + 1);
    for (auto& x : rel) x -= t0;
    g.n_seg = s1 - s0;
    g.h_offsets = rel.data();
    g.d_offsets = a->d_offsets + s0;   // read on the device minus t0
    g.n_tok = T;
    g.k = base + L.k;
    g.v = base + L.v;
    g.beta = has_beta(a->kind) ? reinterpret_cast<const float*>(base + L.beta) : nullptr;
    g.log_alpha = (a->kind == HYPIC_NO_DECAY) ? nullptr
                                              : reinterpret_cast<const float*>(base + L.log_alpha);
    rc = launch_build(&g, out, d_ws, st, t0, s0, sms);
    if (rc == HYPIC_OK && cudaEventRecord(freed[h], st) != cudaSuccess) rc = HYPIC_ERR_CUDA;
  }
  for (int h = 0; h < 2; ++h) {
    cudaEventDestroy(copied[h]);
    cudaEventDestroy(freed[h]);
  }
  return rc;
}

size_t hypic_build_split_scratch_bytes(const hypic_build_args* a, int64_t piece_tokens) {
  if (check_build_args(a) != HYPIC_OK || piece_tokens < 1) return 0;
  const SplitPlan sp = split_plan(a, piece_tokens);
  if (static_cast<int64_t>(sp.n_pieces + 1) * a->n_streams > INT32_MAX) return 0;
  return split_layout(a, sp).bytes;
}

hypic_status hypic_segment_build_split(const hypic_build_args* a, const hypic_cache* out,
                                       int64_t piece_tokens, void* d_scratch,
                                       size_t scratch_bytes, void* stream) {
  hypic_status s = check_build_args(a);
  if (s != HYPIC_OK) return s;
  if ((s = check_cache(a, out)) != HYPIC_OK) return s;
  if ((s = check_device_inputs(a)) != HYPIC_OK) return s;
  if (piece_tokens < 1) return HYPIC_ERR_SHAPE;
  const SplitPlan sp = split_plan(a, piece_tokens);
  if (static_cast<int64_t>(sp.n_pieces + 1) * a->n_streams > INT32_MAX) return HYPIC_ERR_SHAPE;
  const SplitLayout L = split_layout(a, sp);
  if (!d_scratch || !aligned256(d_scratch) || scratch_bytes < L.bytes) return HYPIC_ERR_WORKSPACE;
  int sms = 0;
  if ((s = check_arch(&sms)) != HYPIC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(d_scratch);
  const bool gdn = factored(a->kind);
  const int lw = log_T_width(a->kind, a->dk);
  const int32_t S = a->n_streams;
  auto F = [&](size_t o) { return reinterpret_cast<float*>(base + o); };
  auto I32p = [&](size_t o) { return reinterpret_cast<int32_t*>(base + o); };
  WsHeader* ws_b = reinterpret_cast<WsHeader*>(base + L.ws_b);
  // the build's status word is the call's: clear it first (the pieces' build
  // clears it again, the compose calls clear their own)
  if (cudaMemsetAsync(ws_b, 0, sizeof(WsHeader), st) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (a->n_seg == 0) return HYPIC_OK;
  if (cudaMemcpyAsync(base + L.off, sp.off.data(), sp.off.size() * 8, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(base + L.order, sp.order.data(), sp.order.size() * 4, cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return HYPIC_ERR_CUDA;
  // the pieces' cache: identity unit n_pieces; for the Qhat product, zero S,
  // log T and exponents and identity start states
  if (launch_split_fill(gdn ? F(L.c_q) : nullptr, gdn ? I32p(L.c_e) : nullptr, F(L.c_l), lw,
                        F(L.c_s), static_cast<int64_t>(sp.n_pieces) * S, S, a->dk,
                        gdn ? F(L.eye) : nullptr, static_cast<int64_t>(a->n_seg) * S, st) !=
      cudaSuccess)
    return HYPIC_ERR_CUDA;
  if (gdn && (cudaMemsetAsync(base + L.z_s, 0, L.z_l - L.z_s, st) != cudaSuccess ||
              cudaMemsetAsync(base + L.z_l, 0, L.eye - L.z_l, st) != cudaSuccess))
    return HYPIC_ERR_CUDA;
  // 1. the pieces, built as segments of their own (no seam window)
  hypic_build_args g = *a;
  g.n_seg = sp.n_pieces;
  g.seam_w = 0;
  g.h_offsets = sp.off.data();
  g.d_offsets = reinterpret_cast<const int64_t*>(base + L.off);
  hypic_cache pc{};
  pc.n_seg = sp.n_pieces + 1;
  pc.n_streams = S;
  pc.dk = a->dk;
  pc.dv = a->dv;
  pc.kind = a->kind;
  pc.Qhat = gdn ? F(L.c_q) : nullptr;
  pc.exp2 = gdn ? I32p(L.c_e) : nullptr;
  pc.log_T = F(L.c_l);
  pc.S = F(L.c_s);
  if ((s = launch_build(&g, &pc, ws_b, st, 0, 0, sms)) != HYPIC_OK) return s;
  // 2. S of each segment: its pieces composed in order from zero
  const int32_t* d_order = I32p(L.order);
  s = hypic_compose(&pc, d_order, a->n_seg, sp.n_pos, nullptr, out->S, nullptr, base + L.ws_c1,
                    hypic_compose_workspace_bytes(&pc, a->n_seg, sp.n_pos, 0), stream);
  if (s != HYPIC_OK) return s;
  // 3. the product of the pieces' Qhat (decays and S set to zero), from I
  if (gdn) {
    hypic_cache qc = pc;
    qc.exp2 = I32p(L.z_e);
    qc.log_T = F(L.z_l);
    qc.S = F(L.z_s);
    s = hypic_compose(&qc, d_order, a->n_seg, sp.n_pos, F(L.eye), out->Qhat, nullptr,
                      base + L.ws_c2, hypic_compose_workspace_bytes(&qc, a->n_seg, sp.n_pos, 0),
                      stream);
    if (s != HYPIC_OK) return s;
  }
  // 4. log T and exponents summed over the pieces, Qhat renormalised
  if (launch_split_finish(d_order, sp.n_pos, static_cast<int64_t>(a->n_seg) * S, S, a->dk,
                          F(L.c_l), gdn ? I32p(L.c_e) : nullptr, lw, out->log_T, out->exp2,
                          gdn ? out->Qhat : nullptr, ws_b,
                          reinterpret_cast<const WsHeader*>(base + L.ws_c1),
                          gdn ? reinterpret_cast<const WsHeader*>(base + L.ws_c2) : nullptr,
                          st) != cudaSuccess)
    return HYPIC_ERR_CUDA;
  return HYPIC_OK;
}

static hypic_status check_seam(const hypic_seam_args* sm, int32_t n) {
  if (sm->w < 1 || sm->w > 64) return HYPIC_ERR_SHAPE;
  if (sm->in_dtype != HYPIC_BF16 && sm->in_dtype != HYPIC_F32) return HYPIC_ERR_DTYPE;
  if (sm->kind < HYPIC_GDN || sm->kind > HYPIC_KDA) return HYPIC_ERR_DTYPE;
  if (sm->o_bf16 != 0 && sm->o_bf16 != 1) return HYPIC_ERR_DTYPE;
  if (n > 0 && (!sm->q || !sm->k || !sm->v || !sm->out_o)) return HYPIC_ERR_NULL;
  if (n > 0 && hypic::has_beta(sm->kind) && !sm->beta) return HYPIC_ERR_NULL;
  if (n > 0 && sm->kind != HYPIC_NO_DECAY && !sm->log_alpha) return HYPIC_ERR_NULL;
  if (!hypic::aligned16(sm->q) || !hypic::aligned16(sm->k) || !hypic::aligned16(sm->v))
    return HYPIC_ERR_SHAPE;
  if ((sm->kind == HYPIC_DIAG_DECAY || sm->kind == HYPIC_KDA) && !hypic::aligned16(sm->log_alpha))
    return HYPIC_ERR_SHAPE;
  return HYPIC_OK;
}

hypic_status hypic_compose(const hypic_cache* c, const int32_t* d_order, int32_t n_req,
                           int32_t n_pos, const float* d_state_in, float* d_state_out,
                           const hypic_seam_args* seam, void* d_ws, size_t ws_bytes,
                           void* stream) {
  if (!c) return HYPIC_ERR_NULL;
  if (n_req < 0 || n_pos < 0 || c->n_seg < 0 || c->n_streams < 1) return HYPIC_ERR_SHAPE;
  if (!(c->dk == c->dv && (c->dk == 64 || c->dk == 128))) return HYPIC_ERR_SHAPE;
  if (c->kind < HYPIC_GDN || c->kind > HYPIC_KDA) return HYPIC_ERR_DTYPE;
  const int64_t n = static_cast<int64_t>(n_req) * n_pos;
  if (n_req > 0 && !d_state_out) return HYPIC_ERR_NULL;
  if (n > 0 && (!d_order || !c->S || !c->log_T)) return HYPIC_ERR_NULL;
  if (n > 0 && factored(c->kind) && (!c->Qhat || !c->exp2)) return HYPIC_ERR_NULL;
  if (!aligned16(c->S) || !aligned16(c->Qhat) || !aligned16(d_state_in) ||
      !aligned16(d_state_out))
    return HYPIC_ERR_SHAPE;
  if (n > 0 && c->n_seg == 0) return HYPIC_ERR_INDEX;
  if (seam) {
    if (seam->kind != c->kind) return HYPIC_ERR_DTYPE;   // the seam tokens' family is the cache's
    hypic_status s = check_seam(seam, static_cast<int32_t>(n > 0));
    if (s != HYPIC_OK) return s;
  }
  const ComposeWsLayout wl = compose_ws_layout(c->n_seg, c->n_streams, c->dk, c->dv,
                                               factored(c->kind), n_req, n_pos, seam ? seam->w : 0);
  if (!d_ws || !aligned256(d_ws) || ws_bytes < wl.bytes) return HYPIC_ERR_WORKSPACE;
  hypic_status s = check_arch(nullptr);
  if (s != HYPIC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* ws = static_cast<WsHeader*>(d_ws);
  if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (n_req == 0) return HYPIC_OK;
  ComposeParams p{};
  p.n_req = n_req;
  p.n_pos = n_pos;
  p.n_seg = c->n_seg;
  p.n_streams = c->n_streams;
  p.dk = c->dk;
  p.dv = c->dv;
  // the compose kernels read the cache's form: matrix (GDN, KDA), per-channel
  // decay, or scalar decay (RetNet, Mamba2-style, none)
  p.kind = factored(c->kind) ? HYPIC_GDN
                             : (c->kind == HYPIC_DIAG_DECAY ? HYPIC_DIAG_DECAY : HYPIC_SCALAR_DECAY);
  p.order = d_order;
  p.Qhat = c->Qhat;
  p.exp2 = c->exp2;
  p.log_T = c->log_T;
  p.Sc = c->S;
  p.state_in = d_state_in;
  p.state_out = d_state_out;
  if (seam) {
    p.w = seam->w;
    p.seam_dtype = seam->in_dtype;
    p.seam_kind = seam->kind;
    p.q = seam->q;
    p.k = seam->k;
    p.v = seam->v;
    p.beta = seam->beta;
    p.log_alpha = seam->log_alpha;
    p.out_o = seam->out_o;
    p.o_bf16 = seam->o_bf16;
    if (wl.rec) p.seam_rec = static_cast<uint8_t*>(d_ws) + wl.rec;
  }
  if (wl.qop) {
    p.qop = static_cast<uint8_t*>(d_ws) + wl.qop;
    p.qop_exp = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(d_ws) + wl.qexp);
  }
  p.ws = ws;
  p.spin_limit = current_spin_limit();
  // gated-delta pairs at dk = dv = 128 compose on the tensor cores; the decay
  // families (elementwise) and dk = 64 on CUDA cores
  const cudaError_t e =
      compose_tc_supported(p) ? launch_compose_tc(p, st) : launch_compose(p, st);
  return e == cudaSuccess ? HYPIC_OK : HYPIC_ERR_CUDA;
}

hypic_status hypic_seam_advance(const hypic_seam_args* seam, int32_t n_req, int32_t n_streams,
                                int32_t dk, int32_t dv, float* d_state, void* d_ws,
                                size_t ws_bytes, void* stream) {
  if (!seam) return HYPIC_ERR_NULL;
  if (n_req < 0 || n_streams < 1) return HYPIC_ERR_SHAPE;
  if (!(dk == dv && (dk == 64 || dk == 128))) return HYPIC_ERR_SHAPE;
  hypic_status s = check_seam(seam, n_req);
  if (s != HYPIC_OK) return s;
  if (n_req > 0 && !d_state) return HYPIC_ERR_NULL;
  if (!aligned16(d_state)) return HYPIC_ERR_SHAPE;
  if (!d_ws || !aligned256(d_ws) || ws_bytes < kWsHeaderBytes) return HYPIC_ERR_WORKSPACE;
  s = check_arch(nullptr);
  if (s != HYPIC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* ws = static_cast<WsHeader*>(d_ws);
  if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return HYPIC_ERR_CUDA;
  if (n_req == 0) return HYPIC_OK;
  // A seam window alone is a compose with one position and no cached pair.
  ComposeParams p{};
  p.n_req = n_req;
  p.n_pos = 1;
  p.n_seg = 0;
  p.n_streams = n_streams;
  p.dk = dk;
  p.dv = dv;
  p.kind = -1;  // no pair to compose
  p.state_in = d_state;
  p.state_out = d_state;
  p.w = seam->w;
  p.seam_dtype = seam->in_dtype;
  p.seam_kind = seam->kind;
  p.q = seam->q;
  p.k = seam->k;
  p.v = seam->v;
  p.beta = seam->beta;
  p.log_alpha = seam->log_alpha;
  p.out_o = seam->out_o;
  p.o_bf16 = seam->o_bf16;
  p.ws = ws;
  p.spin_limit = current_spin_limit();
  return launch_compose(p, st) == cudaSuccess ? HYPIC_OK : HYPIC_ERR_CUDA;
}

}  // extern "C"
