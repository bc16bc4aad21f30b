// moe_dispatch_layout_noalloc: the dispatch layout for callers that cannot
// allocate device memory, e.g. a plugin running inside a host engine that
// owns the whole device memory pool and hands it only input and output
// buffers, or a service that forbids cudaMalloc after start-up because an
// allocation can synchronise the device and stall other streams.
//
// It runs the same three layout kernels as moe_dispatch_layout; only the
// scratch differs.  Instead of a caller-provided workspace, the per-chunk
// expert histograms live in the file-scope array below, which every GPU
// that loads this library holds until the process exits.
//
//  - Maximum: ceil(T*k / 2048) * E * 4 bytes must fit in
//    MOE_NOALLOC_LAYOUT_SCRATCH_BYTES (1 MiB); larger requests return
//    MOE_ERR_UNSUPPORTED and launch nothing.
//  - Set-up: the first call on each device, with that device current, looks
//    up the array's device address (cudaGetSymbolAddress) and caches it,
//    keyed by the unique id of the device's current CUDA context.  If that
//    context is destroyed and another created (cudaDeviceReset, or a host
//    engine that resets the device), the module is loaded again and the
//    array may move: the next call sees a new context id and looks the
//    address up again.  Make the first call in each context before any
//    stream capture.
//  - Sharing: every call uses the same array and leaves the last call's
//    histograms in it.  Nothing needs clearing: each call writes every cell
//    it later reads.  Calls whose kernels overlap on the GPU (different
//    streams with no ordering between them) race on the array.
//  - No cudaMalloc, cudaFree or other allocating routine is called.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

static __device__ __align__(256) int32_t
    g_layout_scratch[MOE_NOALLOC_LAYOUT_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  void* ptr;
  unsigned long long ctx_id;   // context the address belongs to
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (cuCtxGetId, never
// reused within a process); false when there is none or the driver lacks
// the call.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<CtxGetCurrentFn>(nullptr);
    }
    return reinterpret_cast<CtxGetCurrentFn>(fn);
  }();
  static CtxGetIdFn get_id = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<CtxGetIdFn>(nullptr);
    }
    return reinterpret_cast<CtxGetIdFn>(fn);
  }();
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current context (nullptr on failure).
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  if (g_scratch[dev].ptr != nullptr && current_context_id(&id) &&
      id == g_scratch[dev].ctx_id)
    return g_scratch[dev].ptr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess) {
    cudaGetLastError();   // leave no pending error behind for the caller
    g_scratch[dev].ptr = nullptr;
    return nullptr;
  }
  // the lookup made the device's primary context current if it was not;
  // without a context id the address is looked up again on every call
  if (current_context_id(&id)) {
    g_scratch[dev].ptr = p;
    g_scratch[dev].ctx_id = id;
  } else {
    g_scratch[dev].ptr = nullptr;
  }
  return p;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_layout_noalloc(
    int32_t T, int32_t k, int32_t E, int32_t R, int32_t capacity,
    const int32_t* topk_idx, int32_t* expert_counts, int32_t* expert_offsets,
    int32_t* dst_row, int32_t* src_pair, int32_t* n_kept, int32_t* n_dropped,
    int32_t* rank_send_counts, int32_t* rank_send_displs, int32_t* status,
    moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > kLayoutMaxE)
    return MOE_ERR_INVALID;
  if (R < 1 || R > E || E % R != 0) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(T) * k > INT32_MAX) return MOE_ERR_INVALID;
  if (expert_counts == nullptr || expert_offsets == nullptr ||
      n_kept == nullptr || n_dropped == nullptr ||
      rank_send_counts == nullptr || rank_send_displs == nullptr)
    return MOE_ERR_INVALID;
  if (T > 0 &&
      (topk_idx == nullptr || dst_row == nullptr || src_pair == nullptr))
    return MOE_ERR_INVALID;
  if (layout_ws_bytes(static_cast<int64_t>(T) * k, E) >
      MOE_NOALLOC_LAYOUT_SCRATCH_BYTES)
    return MOE_ERR_UNSUPPORTED;
  void* scratch = scratch_address();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  return launch_layout(T, k, E, R, capacity, topk_idx, expert_counts,
                       expert_offsets, dst_row, src_pair, n_kept, n_dropped,
                       rank_send_counts, rank_send_displs, scratch, status,
                       reinterpret_cast<cudaStream_t>(stream));
}
