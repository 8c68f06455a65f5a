// Segment build without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need a
// build: a serving loop that must not let cudaMalloc synchronise the device in
// the middle of a request, a host framework whose own allocator owns all device
// memory and forbids allocations from libraries, or an embedding with a fixed
// device-memory budget decided at start-up.  For them this entry point runs
// the same build as hypic_segment_build, with its scratch (status word,
// work-queue counter and LPT work list) in a fixed device array that lives in
// this library for the life of the process.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address (in host code the name denotes a host-side
// stand-in), so the device address is looked up with cudaGetSymbolAddress, with
// the device current.  Outside a stream capture every call looks it up again
// (a device reset unloads the module, so an address kept from before it would
// be stale); a call made while its stream is capturing reuses the address the
// last uncaptured call on that device found.
#include <mutex>

#include "hypic_internal.h"

namespace hypic {
namespace {

constexpr size_t kStaticWsBytes =
    kWsHeaderBytes + static_cast<size_t>(HYPIC_STATIC_WS_MAX_ITEMS) * sizeof(WorkItem);

// Every GPU that loads the library holds these bytes until the process exits.
__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (nullptr on failure).
void* static_ws_address(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (cap != cudaStreamCaptureStatusNone) return g_addr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
  g_addr[dev] = p;
  return p;
}

}  // namespace
}  // namespace hypic

extern "C" hypic_status hypic_segment_build_static_ws(const hypic_build_args* args,
                                                      const hypic_cache* out, void* stream,
                                                      int32_t* h_status) {
  using namespace hypic;
  // the ordinary entry point's host checks first, in its order
  hypic_status s = check_build_call(args, out);
  if (s != HYPIC_OK) return s;
  const int64_t n_items = static_cast<int64_t>(args->n_seg) * args->n_streams;
  if (n_items > HYPIC_STATIC_WS_MAX_ITEMS) return HYPIC_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = static_ws_address(st);
  if (!ws) return HYPIC_ERR_CUDA;
  // The existing build path clears the status word and the queue counter at
  // the start of every call; the work list is rewritten before it is read.
  s = hypic_segment_build(args, out, ws, kStaticWsBytes, stream);
  if (s != HYPIC_OK || !h_status) return s;
  return hypic_read_device_status(ws, stream, h_status);
}
