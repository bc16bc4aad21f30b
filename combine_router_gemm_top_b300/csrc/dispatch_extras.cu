// Dispatch bookkeeping beyond the compact layout.
//
// dispatch matrix  ("All-to-All Communication", the routing simulation
//                  listing and its printed dispatch matrix): pairs sent from
//                  each of n_src equal contiguous token shards (virtual
//                  source devices) to each of n_dst contiguous expert blocks
//                  (virtual destination devices).  Dropped pairs are not
//                  sent.  Integer atomics only, so the result is exact.
// padded layout    ("Expert Parallelism in LLMs", Static Capacity Factors and
//                  Token Dropping: fixed buffers of C_expert rows per expert,
//                  empty slots are padding): the row of each kept pair in an
//                  [E, C, D] buffer, the uniform offsets e*C, and the zero
//                  fill of the padding rows.  moe_permute, moe_grouped_ffn and
//                  moe_combine then run unchanged on the padded rows.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kMatrixThreads = 256;
constexpr int kMatrixPairsPerBlock = 1024;

__global__ void zero_i32_kernel(int32_t* p, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0;
}

// grid (chunks, n_src): block (c, s) counts pairs [c*1024, (c+1)*1024) of
// source shard s into a shared histogram over destinations, then adds it
// to row s of the matrix.  Each warp takes 32 consecutive pairs at a time;
// lanes with the same destination are counted together (one shared atomic
// per distinct destination in the warp).
__global__ void __launch_bounds__(kMatrixThreads)
    dispatch_matrix_kernel(int64_t pairs_per_src, int k, int E, int n_dst,
                           const int32_t* __restrict__ topk_idx,
                           const int32_t* __restrict__ dst_row,
                           int32_t* __restrict__ matrix, int32_t* status) {
  extern __shared__ int32_t hist[];
  for (int i = threadIdx.x; i < n_dst; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.y) * pairs_per_src;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kMatrixPairsPerBlock;
  const int64_t hi = min(pairs_per_src, lo + kMatrixPairsPerBlock);
  const int epr = E / n_dst;
  const int lane = threadIdx.x & 31;
  // q0 is the same on every lane of a warp, so each warp runs whole
  // iterations (the match below needs all 32 lanes)
  for (int64_t q0 = lo + (threadIdx.x & ~31); q0 < hi; q0 += blockDim.x) {
    const int64_t q = q0 + lane;
    int d = -1;
    if (q < hi) {
      const int64_t p = base + q;
      const int32_t row = dst_row != nullptr ? __ldg(dst_row + p) : 0;
      const int e = __ldg(topk_idx + p);
      if (row >= 0) {
        if (e < 0 || e >= E)
          set_status(status, MOE_ERR_INDEX);
        else
          d = e / epr;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    if (d >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
  }
  __syncthreads();
  int32_t* row = matrix + static_cast<int64_t>(blockIdx.y) * n_dst;
  for (int i = threadIdx.x; i < n_dst; i += blockDim.x)
    if (hist[i] != 0) atomicAdd(row + i, hist[i]);
}

moe_status launch_dispatch_matrix(int T, int k, int E, int n_src, int n_dst,
                                  const int32_t* topk_idx,
                                  const int32_t* dst_row, int32_t* matrix,
                                  int32_t* status, cudaStream_t stream) {
  const int64_t cells = static_cast<int64_t>(n_src) * n_dst;
  zero_i32_kernel<<<static_cast<unsigned>(ceil_div(cells, 256)), 256, 0,
                    stream>>>(matrix, cells);
  const int64_t pairs_per_src = static_cast<int64_t>(T / n_src) * k;
  if (pairs_per_src > 0) {
    const dim3 grid(static_cast<unsigned>(ceil_div(pairs_per_src,
                                                   kMatrixPairsPerBlock)),
                    static_cast<unsigned>(n_src));
    dispatch_matrix_kernel<<<grid, kMatrixThreads,
                             static_cast<size_t>(n_dst) * sizeof(int32_t),
                             stream>>>(pairs_per_src, k, E, n_dst, topk_idx,
                                       dst_row, matrix, status);
  }
  return launch_status();
}

// dst_row_padded[p] = e*C + (dst_row[p] - expert_offsets[e]) for a kept
// pair of expert e, -1 for a dropped one; offsets_padded[e] = e*C.
__global__ void padded_layout_kernel(int64_t P, int E, int capacity,
                                     const int32_t* __restrict__ topk_idx,
                                     const int32_t* __restrict__ dst_row,
                                     const int32_t* __restrict__ offsets,
                                     int32_t* __restrict__ dst_row_padded,
                                     int32_t* __restrict__ offsets_padded,
                                     int32_t* status) {
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p <= E) offsets_padded[p] = static_cast<int32_t>(p * capacity);
  if (p >= P) return;
  const int r = __ldg(dst_row + p);
  int out = -1;
  if (r >= 0) {
    const int e = __ldg(topk_idx + p);
    if (e >= 0 && e < E) {
      const int pos = r - __ldg(offsets + e);
      if (pos >= 0 && pos < capacity)
        out = e * capacity + pos;
      else
        set_status(status, MOE_ERR_INDEX);
    } else {
      set_status(status, MOE_ERR_INDEX);
    }
  }
  dst_row_padded[p] = out;
}

moe_status launch_padded_layout(int T, int k, int E, int capacity,
                                const int32_t* topk_idx,
                                const int32_t* dst_row,
                                const int32_t* offsets,
                                int32_t* dst_row_padded,
                                int32_t* offsets_padded, int32_t* status,
                                cudaStream_t stream) {
  const int64_t P = static_cast<int64_t>(T) * k;
  const int64_t n = P > E + 1 ? P : E + 1;
  padded_layout_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                         stream>>>(P, E, capacity, topk_idx, dst_row, offsets,
                                   dst_row_padded, offsets_padded, status);
  return launch_status();
}

// Zero the padding rows [e*C + count_e, (e+1)*C) of every expert: one warp
// per padded row, 16-byte stores; rows holding a kept pair are skipped.
__global__ void __launch_bounds__(256)
    pad_fill_kernel(int64_t rows, int capacity, int nvec,
                    const int32_t* __restrict__ counts,
                    uint4* __restrict__ buf) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * 8;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t r = w0; r < rows; r += nw) {
    const int e = static_cast<int>(r / capacity);
    const int pos = static_cast<int>(r - static_cast<int64_t>(e) * capacity);
    if (pos < __ldg(counts + e)) continue;
    uint4* row = buf + r * nvec;
    for (int v = lane; v < nvec; v += 32) st_v4(row + v, z);
  }
}

moe_status launch_pad_fill(int E, int capacity, int D, int dtype,
                           const int32_t* counts, void* buf,
                           cudaStream_t stream, int num_sms) {
  const int64_t rows = static_cast<int64_t>(E) * capacity;
  if (rows == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const int64_t want = ceil_div(rows, 8);
  const int64_t cap_blocks = static_cast<int64_t>(num_sms) * 8;
  pad_fill_kernel<<<static_cast<unsigned>(want < cap_blocks ? want
                                                            : cap_blocks),
                    256, 0, stream>>>(rows, capacity, nvec, counts,
                                      static_cast<uint4*>(buf));
  return launch_status();
}

}  // namespace moe
