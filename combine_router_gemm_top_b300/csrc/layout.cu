// moe_dispatch_layout kernels: per-expert histogram, exclusive scan with
// the capacity clamp, and the stable per-pair row assignment
// ("Expert Parallelism in LLMs", The Execution Pipeline, step 2 "Local Token
// Permutation"; Static Capacity Factors and Token Dropping: C_expert =
// ceil(CF * k * B * S / E), overflow dropped; "All-to-All Communication",
// expert_parallel_dispatch listing: destination = expert /
// experts_per_device and the bincount of destinations).
//
// Up to 16384 pairs and 256 experts: one block does the whole layout
// (layout_small).  Beyond that, pairs are cut into chunks of 2048 (one block
// each), each chunk into 8 warp sub-chunks of 256.  Three launches:
//   1 layout_hist    per-chunk expert histograms  -> ws[chunk][E]
//   2 layout_scan    (one block) per expert, its chunk column cut into
//                    segments over the block's threads: exclusive prefix
//                    over chunks (in place), totals, capacity clamp,
//                    offsets, rank counts and displacements, n_kept,
//                    n_dropped
//   3 layout_assign  per chunk: per-warp sub-chunk prefixes, then each warp
//                    walks its pairs in order, ranking equal experts inside
//                    a 32-pair step with __match_any_sync; pos = earlier
//                    pairs of the same expert; kept iff pos < capacity.
// All integer: results are identical run to run.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kLayoutWarps = 8;
constexpr int kSubChunk = kLayoutChunk / kLayoutWarps;   // 256

__global__ void __launch_bounds__(256)
    layout_hist_kernel(int64_t P, int E, const int32_t* __restrict__ idx,
                       int32_t* __restrict__ ws, int32_t* status) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kLayoutChunk;
  const int64_t p1 = min(P, p0 + kLayoutChunk);
  bool bad = false;
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = __ldg(idx + p);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&hist[e], 1);
    else
      bad = true;
  }
  if (bad) set_status(status, MOE_ERR_INDEX);
  __syncthreads();
  int32_t* out = ws + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = hist[e];
}

// From the kept count of every expert (shared memory, one block): the
// exclusive scan into offsets, the counts, n_kept, n_dropped, and each
// rank's send count and displacement.  off_s (shared) also receives the
// offsets when not null.
__device__ void layout_finish(int64_t P, int E, int R, const int32_t* kept,
                              int32_t* off_s, int32_t* expert_counts,
                              int32_t* expert_offsets, int32_t* n_kept,
                              int32_t* n_dropped, int32_t* rank_send_counts,
                              int32_t* rank_send_displs) {
  // exclusive scan of kept[0..E): each of 32 lanes of warp 0 scans a
  // contiguous segment, then the segment sums are scanned across lanes
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int seg = (E + 31) / 32;
    const int b = lane * seg;
    const int en = min(E, b + seg);
    int32_t s = 0;
    for (int e = b; e < en; ++e) s += kept[e];
    int32_t incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int32_t run = incl - s;      // exclusive start of this lane's segment
    for (int e = b; e < en; ++e) {
      expert_offsets[e] = run;
      if (off_s != nullptr) off_s[e] = run;
      expert_counts[e] = kept[e];
      run += kept[e];
    }
    if (lane == 31) {
      expert_offsets[E] = incl;
      *n_kept = incl;
      *n_dropped = static_cast<int32_t>(P - incl);
    }
  }
  __syncthreads();
  // rank r owns experts [r*E/R, (r+1)*E/R): its rows are one contiguous run
  const int epr = E / R;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    int32_t start = 0, cnt = 0;
    for (int e = 0; e < r * epr; ++e) start += kept[e];
    for (int e = r * epr; e < (r + 1) * epr; ++e) cnt += kept[e];
    rank_send_counts[r] = cnt;
    rank_send_displs[r] = start;
  }
}

__global__ void __launch_bounds__(1024)
    layout_scan_kernel(int64_t P, int E, int R, int capacity, int nchunks,
                       int32_t* __restrict__ ws, int32_t* expert_counts,
                       int32_t* expert_offsets, int32_t* n_kept,
                       int32_t* n_dropped, int32_t* rank_send_counts,
                       int32_t* rank_send_displs) {
  __shared__ int32_t kept[kLayoutMaxE];
  __shared__ int32_t seg_sum[1024];
  {
    // the chunk column of each expert (E <= 1024) is cut into S = 1024 / E
    // segments; thread (s, e) = (tid / E, tid % E) first adds its segment
    // (independent loads), then rewrites it as the exclusive prefix,
    // starting from the sum of the earlier segments
    const int S = 1024 / E;
    const int seg = (nchunks + S - 1) / S;
    const int e = threadIdx.x % E;
    const int sg = threadIdx.x / E;
    const bool on = sg < S;
    const int c_begin = sg * seg;
    const int c_end = min(nchunks, c_begin + seg);
    int32_t mine = 0;
    if (on) {
#pragma unroll 4
      for (int c = c_begin; c < c_end; ++c)
        mine += ws[static_cast<int64_t>(c) * E + e];
    }
    seg_sum[threadIdx.x] = mine;
    __syncthreads();
    if (on) {
      int32_t run = 0;
      for (int q = 0; q < sg; ++q) run += seg_sum[q * E + e];
      for (int c0 = c_begin; c0 < c_end; c0 += 8) {
        int32_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = c0 + i < c_end ? ws[static_cast<int64_t>(c0 + i) * E + e] : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + i < c_end) ws[static_cast<int64_t>(c0 + i) * E + e] = run;
          run += v[i];
        }
      }
      if (sg == S - 1) kept[e] = capacity > 0 ? min(run, capacity) : run;
    }
  }
  __syncthreads();
  layout_finish(P, E, R, kept, nullptr, expert_counts, expert_offsets, n_kept,
                n_dropped, rank_send_counts, rank_send_displs);
}

__global__ void __launch_bounds__(256)
    layout_assign_kernel(int64_t P, int E, int capacity,
                         const int32_t* __restrict__ idx,
                         const int32_t* __restrict__ ws,
                         const int32_t* __restrict__ expert_offsets,
                         int32_t* __restrict__ dst_row,
                         int32_t* __restrict__ src_pair) {
  extern __shared__ int32_t sm[];
  int32_t* whist = sm;                            // [8][E]
  int32_t* off = sm + kLayoutWarps * E;           // [E]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kLayoutChunk;
  for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) off[e] = expert_offsets[e];
  __syncthreads();
  const int64_t s0 = c0 + static_cast<int64_t>(warp) * kSubChunk;
  const int64_t s1 = min(P, s0 + kSubChunk);
  for (int64_t p = s0 + lane; p < s1; p += 32) {
    const int e = __ldg(idx + p);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&whist[warp * E + e], 1);
  }
  __syncthreads();
  // whist[w][e] <- pairs of expert e before sub-chunk w of this chunk,
  // counting all earlier chunks
  const int32_t* base = ws + static_cast<int64_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = base[e];
    for (int w = 0; w < kLayoutWarps; ++w) {
      const int32_t v = whist[w * E + e];
      whist[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  int32_t* my = whist + warp * E;
  for (int64_t pb = s0; pb < s1; pb += 32) {
    const int64_t p = pb + lane;
    const bool in = p < s1;
    const int e = in ? __ldg(idx + p) : -1;
    const bool valid = in && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    // lanes with the same expert id (invalid lanes get distinct keys)
    const int key = valid ? e : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int32_t pos = 0;
    if (valid) pos = my[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) my[e] += __popc(peers);
    __syncwarp();
    if (in) {
      const bool kept = valid && (capacity <= 0 || pos < capacity);
      const int32_t r = kept ? off[e] + pos : -1;
      dst_row[p] = r;
      if (kept) src_pair[r] = static_cast<int32_t>(p);
    }
  }
}

// The whole layout in one block of 32 warps, for up to kSmallP pairs and
// kSmallE experts.  Warp w owns a contiguous range of pairs (whole 32-pair
// steps); it counts its experts, a prefix over warps gives each warp the
// pairs of each expert before its range, the scan and capacity clamp follow,
// then each warp walks its range in order, ranking equal experts inside a
// 32-pair step with __match_any_sync exactly as layout_assign does.
constexpr int64_t kSmallP = 16384;
constexpr int kSmallE = 256;
constexpr int kSmallWarps = 32;

__global__ void __launch_bounds__(kSmallWarps * 32)
    layout_small_kernel(int64_t P, int E, int R, int capacity,
                        const int32_t* __restrict__ idx,
                        int32_t* expert_counts, int32_t* expert_offsets,
                        int32_t* dst_row, int32_t* src_pair, int32_t* n_kept,
                        int32_t* n_dropped, int32_t* rank_send_counts,
                        int32_t* rank_send_displs, int32_t* status) {
  extern __shared__ int32_t sm[];
  int32_t* whist = sm;                          // [32][E]
  int32_t* kept = sm + kSmallWarps * E;         // [E]
  int32_t* off = kept + E;                      // [E]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int64_t span = ceil_div(ceil_div(P, kSmallWarps), 32) * 32;
  const int64_t s0 = static_cast<int64_t>(warp) * span;
  const int64_t s1 = min(P, s0 + span);
  bool bad = false;
  for (int64_t p = s0 + lane; p < s1; p += 32) {
    const int e = __ldg(idx + p);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicAdd(&whist[warp * E + e], 1);
    else
      bad = true;
  }
  if (bad) set_status(status, MOE_ERR_INDEX);
  __syncthreads();
  // whist[w][e] <- pairs of expert e before warp w's range; kept = clamp
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int32_t v = whist[w * E + e];
      whist[w * E + e] = run;
      run += v;
    }
    kept[e] = capacity > 0 ? min(run, capacity) : run;
  }
  __syncthreads();
  layout_finish(P, E, R, kept, off, expert_counts, expert_offsets, n_kept,
                n_dropped, rank_send_counts, rank_send_displs);
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  int32_t* my = whist + warp * E;
  for (int64_t pb = s0; pb < s1; pb += 32) {
    const int64_t p = pb + lane;
    const bool in = p < s1;
    const int e = in ? __ldg(idx + p) : -1;
    const bool valid = in && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    // lanes with the same expert id (invalid lanes get distinct keys)
    const int key = valid ? e : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int32_t pos = 0;
    if (valid) pos = my[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) my[e] += __popc(peers);
    __syncwarp();
    if (in) {
      const bool kept_p = valid && (capacity <= 0 || pos < capacity);
      const int32_t r = kept_p ? off[e] + pos : -1;
      dst_row[p] = r;
      if (kept_p) src_pair[r] = static_cast<int32_t>(p);
    }
  }
}

int layout_launches(int64_t P, int E) {
  if (P <= kSmallP && E <= kSmallE) return 1;
  return P > 0 ? 3 : 1;
}

size_t layout_ws_bytes(int64_t P, int E) {
  const int64_t nchunks = ceil_div(P, kLayoutChunk);
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * E * sizeof(int32_t);
}

moe_status launch_layout(int T, int k, int E, int R, int capacity,
                         const int32_t* topk_idx, int32_t* expert_counts,
                         int32_t* expert_offsets, int32_t* dst_row,
                         int32_t* src_pair, int32_t* n_kept,
                         int32_t* n_dropped, int32_t* rank_send_counts,
                         int32_t* rank_send_displs, void* ws, int32_t* status,
                         cudaStream_t stream) {
  const int64_t P = static_cast<int64_t>(T) * k;
  if (P <= kSmallP && E <= kSmallE) {
    const size_t smem = static_cast<size_t>(kSmallWarps + 2) * E * sizeof(int32_t);
    layout_small_kernel<<<1, kSmallWarps * 32, smem, stream>>>(
        P, E, R, capacity, topk_idx, expert_counts, expert_offsets, dst_row,
        src_pair, n_kept, n_dropped, rank_send_counts, rank_send_displs,
        status);
    return launch_status();
  }
  const int nchunks = static_cast<int>(ceil_div(P, kLayoutChunk));
  int32_t* w = static_cast<int32_t*>(ws);
  if (nchunks > 0)
    layout_hist_kernel<<<nchunks, 256, E * sizeof(int32_t), stream>>>(
        P, E, topk_idx, w, status);
  layout_scan_kernel<<<1, 1024, 0, stream>>>(
      P, E, R, capacity, nchunks, w, expert_counts, expert_offsets, n_kept,
      n_dropped, rank_send_counts, rank_send_displs);
  if (nchunks > 0) {
    const size_t smem = (kLayoutWarps + 1) * E * sizeof(int32_t);
    static std::atomic<uint64_t> attr_done{0};
    if (!set_smem_limit_once(reinterpret_cast<const void*>(layout_assign_kernel),
                             (kLayoutWarps + 1) * kLayoutMaxE * 4, &attr_done))
      return MOE_ERR_CUDA;
    layout_assign_kernel<<<nchunks, 256, smem, stream>>>(
        P, E, capacity, topk_idx, w, expert_offsets, dst_row, src_pair);
  }
  return launch_status();
}

}  // namespace moe
