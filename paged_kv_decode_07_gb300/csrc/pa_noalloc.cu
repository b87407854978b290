// pa_noalloc.cu -- pa_decode_noalloc: paged decode for callers that cannot
// allocate device memory.
//
// pa_decode needs a caller-provided device workspace (the split-K plan and
// the fp32 partial results).  Some callers cannot obtain one: code running
// inside a framework that owns every device allocation through its own
// pool, plugins and custom operators that are handed only input and output
// buffers, and hosts that forbid cudaMalloc after start-up.  For them this
// file keeps the workspace in a file-scope device array of fixed size,
// PA_NOALLOC_SCRATCH_BYTES (16 MiB).  Every GPU that loads this library
// holds that array until the process exits.
//
// Host code must not pass `g_scratch` itself to a kernel: on the host the
// name is only a stand-in for the device symbol.  The first call on each
// device (with that device current) resolves the real device address with
// cudaGetSymbolAddress and caches it; that first call should therefore come
// before any stream capture.  The cached address belongs to the device's
// current primary context: after cudaDeviceReset (or any teardown of that
// context) the module is loaded afresh at another address, so a process
// that resets a device must not call this entry point on it again.  No call
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
//
// All calls share the one array and it keeps the previous call's contents.
// Nothing in it has to start at zero (the planner rewrites the header, the
// work list and every partial it later reads on each call), but two calls
// whose work can overlap on the GPU (different streams without ordering, or
// different host threads) race on it and give wrong results.
#include <mutex>

#include "pa_internal.cuh"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// device address of g_scratch on the current device (set up once per device)
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(const pa_kv_cache *kv, const pa_problem *prob,
                                 pa_stream_t stream) {
  pa_options opt;
  opt.kernel = 0;
  opt.split_blocks = 0;
  opt.target_items = pa::kDefaultTargetItems;
  opt.event_begin = nullptr;
  opt.event_end = nullptr;
  opt.test_flags = 0;
  // pa_decode validates the arguments and the workspace size (returning its
  // own status codes, with nothing launched, when either is wrong)
  void *ws = nullptr;
  const int st = scratch_address(&ws);
  if (st != PA_OK) return st;
  return pa_decode(kv, prob, &opt, ws, kScratchBytes, stream);
}
