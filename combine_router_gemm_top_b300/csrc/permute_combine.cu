// moe_permute and moe_combine: the two HBM-bound row movers around the
// expert GEMMs.
//
// permute  ("Expert Parallelism in LLMs", The Execution Pipeline, step 2:
//           tokens physically reordered into contiguous per-destination
//           buffers) -- token-major scatter: each token row is read from
//           HBM once and written to each kept destination row, so the
//           traffic is T*D*s read + N*D*s written.
// combine  (same page, step 6 "Unpermutation and Weighted Reduction") --
//           token-major gather: y[t] = sum_j g[t,j] * yp[dst_row[t*k+j]],
//           fp32 accumulation in slot order (deterministic, no atomics),
//           traffic N*D*s read + T*D*s written.
//
// One warp per token; each lane moves 16-byte vectors.  Up to 4 vectors
// per lane are in flight per step for memory-level parallelism.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRowWarps = 8;   // warps per block
constexpr int kUnroll = 4;     // 16-byte vectors per lane per step

template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
    permute_kernel(int64_t n_tok, int k, int nvec, const uint4* __restrict__ x,
                   const int32_t* __restrict__ dst_row, uint4* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  for (int64_t t = warp_g; t < n_tok; t += nwarps) {
    // lane j < k holds the destination row of slot j
    const int32_t my_dst = lane < k ? __ldg(dst_row + t * k + lane) : -1;
    const uint4* src = x + t * nvec;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * 32;
        if (v < nvec) buf[u] = ld_nc_v4(src + v);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_dst, j);
        if (r < 0) continue;
        uint4* dst = xp + static_cast<int64_t>(r) * nvec;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32;
          if (v < nvec) st_v4(dst + v, buf[u]);
        }
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
    combine_kernel(int64_t n_tok, int k, int nvec, const uint4* __restrict__ yp,
                   const int32_t* __restrict__ dst_row,
                   const float* __restrict__ gate, uint4* __restrict__ y) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  for (int64_t t = warp_g; t < n_tok; t += nwarps) {
    const int32_t my_dst = lane < k ? __ldg(dst_row + t * k + lane) : -1;
    // gate == nullptr: unit gates (the permute backward sums the rows)
    const float my_g =
        lane < k ? (gate != nullptr ? __ldg(gate + t * k + lane) : 1.0f)
                 : 0.0f;
    uint4* out = y + t * nvec;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
      float acc[kUnroll][N];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int i = 0; i < N; ++i) acc[u][i] = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_dst, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (r < 0) continue;
        const uint4* src = yp + static_cast<int64_t>(r) * nvec;
        uint4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32;
          if (v < nvec) buf[u] = ld_nc_v4(src + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          float f[N];
          Vec16<T>::to_f32(buf[u], f);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[u][i] = fmaf(g, f[i], acc[u][i]);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * 32;
        if (v < nvec) st_v4(out + v, Vec16<T>::from_f32(acc[u]));
      }
    }
  }
}

static unsigned row_grid(int64_t T, int num_sms) {
  // enough resident warps to cover HBM latency: 8 blocks of 8 warps per SM
  const int64_t want = ceil_div(T, kRowWarps);
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<unsigned>(want < cap ? want : cap);
}

moe_status launch_permute(int T, int k, int D, int dtype, const void* x,
                          const int32_t* dst_row, void* xp,
                          cudaStream_t stream, int num_sms) {
  if (T == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const unsigned grid = row_grid(T, num_sms);
  if (dtype == MOE_BF16)
    permute_kernel<__nv_bfloat16><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(x), dst_row,
        static_cast<uint4*>(xp));
  else
    permute_kernel<float><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(x), dst_row,
        static_cast<uint4*>(xp));
  return launch_status();
}

moe_status launch_combine(int T, int k, int D, int dtype, const void* yp,
                          const int32_t* dst_row, const float* gate, void* y,
                          cudaStream_t stream, int num_sms) {
  if (T == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const unsigned grid = row_grid(T, num_sms);
  if (dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(yp), dst_row, gate,
        static_cast<uint4*>(y));
  else
    combine_kernel<float><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(yp), dst_row, gate,
        static_cast<uint4*>(y));
  return launch_status();
}

}  // namespace moe
