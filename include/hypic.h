/*
 * hypic.h -- C ABI of libhypic.so: position-independent caching of
 * linear-attention state on one GB300 (sm_103a) GPU.
 *
 * What the library computes (HYPIC; youleyou.com article "小红书联合北大上交提出
 * HYPIC，位置无关缓存降低首token延迟3.25倍", linear-layer paragraph, and the
 * llm-wiki summary "HYPIC: 하이브리드 어텐션 LLM 서빙에서 포지션 독립적 캐싱으로 TTFT를
 * 2.45배 낮추는 방법", section "세그먼트 누적 전이 연산자"):
 *
 *   per token t of a stream (one linear layer x head):
 *     S_t = A_t S_{t-1} + b_t k_t v_t^T            S is dk x dv, left-multiplied
 *     gated delta (GDN):  A_t = alpha_t (I - beta_t k_t k_t^T),  b_t = beta_t
 *     RetNet (scalar):    A_t = gamma I,                         b_t = 1
 *     GLA (diagonal):     A_t = diag(alpha_t) on the key axis,   b_t = 1
 *     plain:              A_t = I,                               b_t = 1
 *     Mamba2 (token):     A_t = alpha_t I, alpha_t per token,    b_t = 1
 *     KDA:                A_t = (I - beta_t k_t k_t^T) diag(alpha_t),  b_t = beta_t
 *     alpha_t = exp(g_t), g_t = log(alpha_t) is the fp32 input ("log_alpha").
 *   (The pages name Mamba2 and KDA only; their updates follow the Mamba2 paper,
 *   "Transformers are SSMs", state space duality section, and the Kimi Linear
 *   paper, KDA section.)
 *   segment C of L tokens:  T_C = A_L ... A_1,  S(C|0) = S_L from S_0 = 0;
 *   composition:            S(C1 C2) = T(C2) S(C1) + S(C2).
 *
 * Seam window (same article, seam-window paragraph): the first w tokens of a
 * segment are not cached; at reuse they are advanced token by token under the
 * full prefix and each emits o_t = S_t^T q_t for the attention layer above.
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer.  The library allocates no device memory,
 *    creates no streams and no threads.  Device pointers are plain CUDA device
 *    addresses on the current device; host pointers are ordinary host memory.
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued asynchronously on it.
 *  - Everything checkable on the host is checked before any launch; a call
 *    that returns an error has launched nothing.
 *  - Errors a kernel detects (an order index out of range, a bounded wait that
 *    ran out) are written to a status word in the caller's workspace; only
 *    hypic_read_device_status synchronises.  Each launching call clears that
 *    word first, so read it before reusing the workspace.
 *  - Nothing aborts: no exit, abort, trap or device assert.
 *  - Supported: dk = dv in {64, 128}; k/v/q dtype bf16 or fp32; arch sm_103
 *    (anything else returns HYPIC_ERR_ARCH).
 *  - Outputs are bitwise deterministic run to run.
 */
#ifndef HYPIC_H
#define HYPIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hypic_status {
  HYPIC_OK = 0,
  HYPIC_ERR_NULL = 1,           /* a required pointer is NULL */
  HYPIC_ERR_SHAPE = 2,          /* unsupported dk/dv/w/count */
  HYPIC_ERR_OFFSETS = 3,        /* offsets[0] != 0, decreasing, or last != n_tok */
  HYPIC_ERR_INDEX = 4,          /* an order index outside [0, n_seg) */
  HYPIC_ERR_DTYPE = 5,          /* unsupported dtype / kind combination */
  HYPIC_ERR_WORKSPACE = 6,      /* workspace NULL, misaligned or too small */
  HYPIC_ERR_ARCH = 7,           /* current device is not sm_103 */
  HYPIC_ERR_CUDA = 8,           /* a CUDA runtime/driver call failed */
  HYPIC_ERR_DEVICE_TIMEOUT = 9  /* a bounded device wait ran out */
} hypic_status;

typedef enum hypic_kind {
  HYPIC_GDN = 0,           /* gated delta rule */
  HYPIC_SCALAR_DECAY = 1,  /* RetNet: per-stream constant gamma */
  HYPIC_DIAG_DECAY = 2,    /* GLA: per-token, per-key-channel alpha */
  HYPIC_NO_DECAY = 3,      /* plain linear attention */
  HYPIC_TOKEN_DECAY = 4,   /* Mamba2-style: per-token scalar alpha */
  HYPIC_KDA = 5            /* KDA: gated delta rule with a per-key-channel gate */
} hypic_kind;

typedef enum hypic_dtype { HYPIC_BF16 = 0, HYPIC_F32 = 1 } hypic_dtype;

/* Inputs of one build call: n_seg segments packed varlen, n_streams streams
 * (layers x heads flattened) of one kind.
 *   h_offsets  host int64 [n_seg+1]; offsets[0] = 0, non-decreasing,
 *              offsets[n_seg] = n_tok, n_tok < 2^31 (HYPIC_ERR_SHAPE otherwise:
 *              token coordinates are 32-bit on the device).  Segment i is tokens
 *              [offsets[i], offsets[i+1]); its cached BODY skips the first
 *              min(seam_w, L_i) tokens (the seam window).  Validated on the
 *              host before any launch.
 *   d_offsets  device int64 [n_seg+1] holding the same values; the device
 *              derives the LPT-ordered work list from it (no host-to-device
 *              copy, no synchronisation).  A device copy that is not a valid
 *              offsets array sets HYPIC_ERR_OFFSETS in the status word.
 *   k          device [n_tok][n_streams][dk], in_dtype
 *   v          device [n_tok][n_streams][dv], in_dtype
 *   beta       device fp32 [n_tok][n_streams]; GDN and KDA (NULL otherwise)
 *   log_alpha  device fp32; GDN, TOKEN [n_tok][n_streams]; DIAG, KDA
 *              [n_tok][n_streams][dk]; SCALAR [n_streams] (log gamma per
 *              stream); NO_DECAY: NULL.
 * The device arrays k, v and (DIAG, KDA) log_alpha, like the cache's Qhat and
 * S, start on a 16-byte boundary (the kernels read them by TMA and 16-byte
 * vector loads); otherwise the call returns HYPIC_ERR_SHAPE before any launch.
 * The host-input entry stages its inputs into aligned device buffers, so only
 * its cache is held to this. */
typedef struct hypic_build_args {
  int32_t n_seg;
  int32_t seam_w;
  int32_t n_streams;
  int32_t dk;
  int32_t dv;
  int32_t kind;      /* hypic_kind */
  int32_t in_dtype;  /* hypic_dtype of k and v */
  int32_t reserved0;
  int64_t n_tok;
  const int64_t* h_offsets;
  const int64_t* d_offsets;
  const void* k;
  const void* v;
  const float* beta;
  const float* log_alpha;
} hypic_build_args;

/* The cache: one (T_C, S(C|0)) pair per (segment, stream), device memory.
 * Unit u = seg * n_streams + stream.
 *   GDN, KDA: T = exp(log_T[u]) * 2^exp2[u] * Qhat[u]   (decay and scale
 *           factored out so long segments stay representable in fp32);
 *           Qhat fp32 [n_seg][n_streams][dk][dk] row-major, exp2 int32
 *           [n_seg][n_streams], log_T fp32 [n_seg][n_streams].  For KDA,
 *           log_T is the sum over the body of each token's largest log-gate
 *           (the slowest channel) and Qhat carries the rest of the gates.
 *   SCALAR, TOKEN, NO_DECAY: T = exp(log_T[u]) I; log_T fp32
 *           [n_seg][n_streams]; Qhat, exp2 unused (may be NULL).
 *   DIAG:   T = diag(exp(log_T[u][:])); log_T fp32 [n_seg][n_streams][dk].
 *   S       fp32 [n_seg][n_streams][dk][dv] row-major (S[i][j], i = key index).
 * A segment whose body is empty holds the identity pair (Qhat = I, exp2 = 0,
 * log_T = 0, S = 0). */
typedef struct hypic_cache {
  int32_t n_seg;
  int32_t n_streams;
  int32_t dk;
  int32_t dv;
  int32_t kind;
  int32_t reserved0;
  float* Qhat;
  int32_t* exp2;
  float* log_T;
  float* S;
} hypic_cache;

/* Seam-window tokens for n_req requests x n_pos positions, advanced with the
 * transitions of family `kind` (zero = gated delta):
 *   q, k  device [n_req][n_pos][w][n_streams][dk], in_dtype
 *   v     device [n_req][n_pos][w][n_streams][dv], in_dtype
 *   beta  device fp32 [n_req][n_pos][w][n_streams]; GDN and KDA (else unused)
 *   log_alpha device fp32; GDN, TOKEN [n_req][n_pos][w][n_streams]; DIAG, KDA
 *         [n_req][n_pos][w][n_streams][dk]; SCALAR [n_streams] (log gamma per
 *         stream, as in the build); NO_DECAY unused
 *   out_o device [n_req][n_pos][w][n_streams][dv], fp32 or (o_bf16) bf16:
 *         o_t = S_t^T q_t read after token t's update. */
typedef struct hypic_seam_args {
  int32_t w;
  int32_t in_dtype;
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* log_alpha;
  void* out_o;
  int32_t kind;       /* hypic_kind of the tokens' transitions */
  int32_t o_bf16;     /* 0: out_o fp32; 1: out_o bf16 (rounded to nearest even) */
} hypic_seam_args;

/* Bytes of device workspace a build call needs (256-byte aligned buffer). */
size_t hypic_build_workspace_bytes(const hypic_build_args* args);

/* Segment build: for every (segment, stream) unit, the pair (T_C, S(C|0)) of
 * its body (youleyou.com article, linear-layer paragraph: cache the pair at a
 * segment's first prefill).  Work items are ordered longest body first
 * (segment-parallelism paragraph: LPT balancing) and taken from a device
 * queue by persistent CTAs.  GDN and KDA with bf16 k/v at dk = dv = 128 run
 * chunked tensor-core builds; fp32 k/v, dk = 64 and the decay families run
 * their own kernels.  The KDA tensor-core build takes each 64-token chunk's
 * decay from its start; a unit with a chunk in which some key channel decays
 * by more than e^-64 relative to the token-wise largest gate is rebuilt by the
 * token recurrence in the same call (same stream, same results layout).
 * Errors: NULL, SHAPE, OFFSETS, DTYPE, WORKSPACE, ARCH, CUDA. */
hypic_status hypic_segment_build(const hypic_build_args* args, const hypic_cache* out,
                                 void* d_ws, size_t ws_bytes, void* stream);

/* Segment build from HOST-resident inputs with the copies overlapped with the
 * build (the same pairs as hypic_segment_build, written into the same cache).
 * Not in the pages: a delivery path for inputs that sit in host memory.
 *  - args: as for hypic_segment_build, except that k, v, beta and log_alpha are
 *    HOST pointers (page-locked memory gives full copy bandwidth; other host
 *    memory works but its copies do not overlap).  h_offsets is read on the
 *    host, d_offsets (the same offsets, device) by the device.
 *  - The segments are taken in groups of consecutive segments of at most
 *    max_group_tokens tokens (a longer segment forms its own group).  Group g's
 *    inputs are copied on copy_stream into one half of d_stage while group g-1
 *    builds on `stream` from the other half; a group's inputs are one
 *    contiguous range of every input array, so each is a single copy.
 *  - d_stage: device buffer of hypic_build_host_stage_bytes(args,
 *    max_group_tokens) bytes (256-byte aligned), owned by the caller and not in
 *    use by other work while the call's operations run.
 *  - d_ws, ws_bytes: as for hypic_segment_build (one workspace, reused by the
 *    groups in order on `stream`).
 *  - Ordering: the copies start after the work already queued on `stream`; the
 *    last build is queued on `stream`, so synchronising `stream` covers the call.
 *    copy_stream may equal `stream` (no overlap).
 * Errors: as hypic_segment_build; WORKSPACE also for a missing or small d_stage. */
size_t hypic_build_host_stage_bytes(const hypic_build_args* args, int64_t max_group_tokens);
hypic_status hypic_segment_build_host(const hypic_build_args* args, const hypic_cache* out,
                                      int64_t max_group_tokens, void* d_stage,
                                      size_t stage_bytes, void* d_ws, size_t ws_bytes,
                                      void* stream, void* copy_stream);

/* Split build of long segments (not in the pages' text as an API; it applies
 * their composition law).  Every segment body is cut into pieces of at most
 * piece_tokens tokens that are built in parallel as pairs of their own; each
 * segment's pair is then the ordered composition of its pieces' pairs:
 * S(C) by composing the pieces from zero, T(C) factored as the summed log T and
 * exponents times the product of the pieces' Qhat (renormalised by a power of
 * two).  Same arguments, outputs and errors as hypic_segment_build; the
 * composition runs through the compose kernels (about fp32 accuracy), so the
 * result equals the unsplit build to within the build's own rounding.
 *  - d_scratch: device buffer of hypic_build_split_scratch_bytes(args,
 *    piece_tokens) bytes (256-byte aligned), owned by the caller; it holds the
 *    pieces' pairs, the work lists and the workspaces.  The call's device status
 *    is read with hypic_read_device_status(d_scratch, ...).
 * Returns 0 bytes for invalid args. */
size_t hypic_build_split_scratch_bytes(const hypic_build_args* args, int64_t piece_tokens);
hypic_status hypic_segment_build_split(const hypic_build_args* args, const hypic_cache* out,
                                       int64_t piece_tokens, void* d_scratch,
                                       size_t scratch_bytes, void* stream);

/* Bytes of device workspace (256-byte aligned) a hypic_compose call over
 * n_req x n_pos positions of `cache` needs, seam_w being the seam window's
 * length (0 without a seam); 0 for a NULL cache.  A 256-byte header (the
 * device status word); for a gated-delta or KDA cache at dk = dv = 128 also
 *  - with seam_w > 0: one 16,896-byte record per (request, position, 8-token
 *    chunk of the window, stream) that the compose fills with the
 *    state-independent part of each seam chunk before the chain runs (about
 *    2.1 KB per seam token-stream);
 *  - when n_req * n_pos >= 2 * n_seg (each pair reused twice or more on
 *    average): a 64 KB copy of every pair's Qhat in the tensor cores' operand
 *    format, made once per call, plus 4 bytes per pair.
 * hypic_seam_advance needs the header only (256 bytes). */
size_t hypic_compose_workspace_bytes(const hypic_cache* cache, int32_t n_req, int32_t n_pos,
                                     int32_t seam_w);

/* Compose cached pairs in request order (youleyou.com article, linear-layer
 * paragraph: reuse by left-multiplying T_C and adding; llm-wiki section
 * "세그먼트 누적 전이 연산자": e_ABC = T_C (T_B e_A + e_B) + e_C):
 * for each request r and stream s, for j = 0 .. n_pos-1,
 *   [if seam != NULL: advance the w seam tokens of (r, j) -- seam-window
 *    paragraph -- emitting o]  then  S <- T_{order[r][j]} S + S_{order[r][j]}.
 *   d_order     device int32 [n_req][n_pos], values in [0, cache->n_seg)
 *               (checked on the device: HYPIC_ERR_INDEX in the status word,
 *               the bad position is skipped)
 *   (the cache's Qhat and S, the states and the seam tokens' q, k, v and, for
 *   DIAG and KDA, log_alpha start on a 16-byte boundary: HYPIC_ERR_SHAPE
 *   otherwise)
 *   d_state_in  device fp32 [n_req][n_streams][dk][dv] or NULL (zero start)
 *   d_state_out device fp32 [n_req][n_streams][dk][dv]; may equal d_state_in
 *   seam        NULL, or the seam tokens of every (r, j), seam->kind equal to
 *               the cache's kind
 * A KDA cache composes through the same matrix form as GDN; a TOKEN cache as
 * the scalar families. 
 * Errors: NULL, SHAPE, DTYPE, WORKSPACE, ARCH, CUDA. */
hypic_status hypic_compose(const hypic_cache* cache, const int32_t* d_order, int32_t n_req,
                           int32_t n_pos, const float* d_state_in, float* d_state_out,
                           const hypic_seam_args* seam, void* d_ws, size_t ws_bytes,
                           void* stream);

/* Advance running states through one seam window per request (seam arrays
 * with n_pos = 1), emitting o_t (youleyou.com article, seam-window paragraph).
 *   d_state device fp32 [n_req][n_streams][dk][dv], updated in place.
 * Errors: NULL, SHAPE, DTYPE, WORKSPACE, ARCH, CUDA. */
hypic_status hypic_seam_advance(const hypic_seam_args* seam, int32_t n_req, int32_t n_streams,
                                int32_t dk, int32_t dv, float* d_state, void* d_ws,
                                size_t ws_bytes, void* stream);

/* Segment build for callers that cannot allocate device memory.  The paper
 * has no counterpart to this entry point; it exists for callers such as a
 * serving loop that must not let cudaMalloc synchronise the device mid-request,
 * a host framework whose allocator owns all device memory, or an embedding with
 * a device-memory budget fixed at start-up.
 * Same computation, arguments and errors as hypic_segment_build, but the
 * scratch (status word, queue counter, work list) lives in a fixed device array
 * inside the library: HYPIC_STATIC_WS_MAX_ITEMS work items (16 bytes each) plus
 * a 256-byte header, 4 MiB + 256 bytes, held on every GPU that loads the library
 * until the process exits.  n_seg * n_streams above the maximum returns
 * HYPIC_ERR_WORKSPACE before any launch.  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 *  - Errors are checked in the order hypic_segment_build checks them (NULL,
 *    SHAPE, DTYPE, OFFSETS, then ARCH); the size limit (WORKSPACE) comes after.
 *  - A call made outside a stream capture looks up the array's device address
 *    (cudaGetSymbolAddress) with the stream's device current, so the address
 *    is fresh after a device reset.  A call made while `stream` is capturing
 *    reuses the address of the last uncaptured call on that device (and
 *    returns HYPIC_ERR_CUDA if there was none): make one call before any
 *    stream capture.
 *  - Every call shares the one array per device: calls whose work overlaps on
 *    the GPU (different streams, or threads without ordering) race.  Calls
 *    enqueued in order on one stream are safe; each call clears the status word
 *    and the queue counter and rewrites the work list before use.
 *  - h_status: NULL, or receives the device status word after the call has
 *    synchronised `stream` (as hypic_read_device_status does). */
#define HYPIC_STATIC_WS_MAX_ITEMS 262144
hypic_status hypic_segment_build_static_ws(const hypic_build_args* args, const hypic_cache* out,
                                           void* stream, int32_t* h_status);

/* Host only.  LPT order of the (segment, stream) items of a build and their
 * greedy static assignment to n_workers workers (youleyou.com article,
 * segment-parallelism paragraph).  Cost of an item = body length
 * L_i - min(seam_w, L_i); order by (-cost, segment, stream); each item in that
 * order goes to the least-loaded worker, lowest id on ties.
 *   h_order  host int32 [n_seg*n_streams]: item ids (seg*n_streams+stream)
 *   h_worker host int32 [n_seg*n_streams] or NULL: worker of item id
 * Errors: NULL, SHAPE, OFFSETS. */
hypic_status hypic_lpt_schedule(const int64_t* h_offsets, int32_t n_seg, int32_t seam_w,
                                int32_t n_streams, int32_t n_workers, int32_t* h_order,
                                int32_t* h_worker);

/* Host only.  offsets[0] = 0, offsets[i+1] = offsets[i] + len[i].
 * Errors: NULL, SHAPE (a negative length or n < 0). */
hypic_status hypic_offsets_from_lengths(const int64_t* h_len, int32_t n, int64_t* h_offsets);

/* Synchronises `stream`, then reads the status word of a workspace.
 * *h_status receives a hypic_status value (HYPIC_OK when no device error). */
hypic_status hypic_read_device_status(const void* d_ws, void* stream, int32_t* h_status);

/* Upper bound on polling iterations of every bounded device wait (mbarrier
 * waits).  0 restores the default.  A wait that runs out sets
 * HYPIC_ERR_DEVICE_TIMEOUT, drains its own copies in flight, frees its tensor
 * memory and returns.  HYPIC_SPIN_EXPIRE_NOW makes every bounded wait give up
 * without polling (a test hook for that error path).  Process-wide; returns the
 * previous value. */
#define HYPIC_SPIN_EXPIRE_NOW 0xFFFFFFFFu
uint32_t hypic_set_spin_limit(uint32_t limit);

/* Order in which a build hands out its (segment, stream) work items to the
 * persistent CTAs: HYPIC_ORDER_LPT, longest body first (the default; youleyou.com
 * article, segment-parallelism paragraph), or HYPIC_ORDER_INDEX, segment order
 * (kept for measuring what the LPT order gains).  The cached pairs are the
 * same either way.  Process-wide; returns the previous order, or -1 (order
 * unchanged) for any other value. */
#define HYPIC_ORDER_LPT 0
#define HYPIC_ORDER_INDEX 1
int32_t hypic_set_build_order(int32_t order);

/* Human-readable name of a status code (static storage). */
const char* hypic_status_str(hypic_status s);

/* Library version as an integer (major*10000 + minor*100 + patch). */
int32_t hypic_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HYPIC_H */
