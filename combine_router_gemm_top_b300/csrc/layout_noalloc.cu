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
//    up the array's device address (cudaGetSymbolAddress) and caches it.
//    Make that first call before any stream capture.
//  - Sharing: every call uses the same array and leaves the last call's
//    histograms in it.  Nothing needs clearing: each call writes every cell
//    it later reads.  Calls whose kernels overlap on the GPU (different
//    streams with no ordering between them) race on the array.
//  - No cudaMalloc, cudaFree or other allocating routine is called.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

static __device__ __align__(256) int32_t
    g_layout_scratch[MOE_NOALLOC_LAYOUT_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device (nullptr on failure).
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess) {
      cudaGetLastError();   // leave no pending error behind for the caller
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
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
