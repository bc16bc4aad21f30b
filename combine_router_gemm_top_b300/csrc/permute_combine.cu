// moe_permute and moe_combine: the two HBM-bound row movers around the
// expert GEMMs.
//
// permute  ("Expert Parallelism in LLMs", The Execution Pipeline, step 2:
//           tokens physically reordered into contiguous per-destination
//           buffers) -- token-major scatter: each token row with a kept
//           slot is read from HBM once and written to each kept destination
//           row, so the traffic is T_kept*D*s read + N*D*s written (T_kept:
//           tokens with at least one kept slot).
// combine  (same page, step 6 "Unpermutation and Weighted Reduction") --
//           token-major gather: y[t] = sum_j g[t,j] * yp[dst_row[t*k+j]],
//           fp32 accumulation in slot order (deterministic, no atomics),
//           traffic N*D*s read + T*D*s written.
//
// One warp per (token, row segment); each lane moves 16-byte vectors, up
// to 4 in flight per step for memory-level parallelism (for a bf16 combine
// with k = 2, 4 per slot, both slots in one round trip).  Row ids at or past
// the buffer's max_rows are skipped (never read or written) and reported as
// MOE_ERR_INDEX.  A row is one segment unless there are too few tokens to
// keep HBM busy: then it is cut into up to 4 segments of at least 128
// vectors, each its own warp (for combine only with k <= 4).
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRowWarps = 8;   // warps per block
constexpr int kUnroll = 4;     // 16-byte vectors per lane per step

template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
    permute_kernel(int64_t n_tok, int k, int nvec, int nseg,
                   const uint4* __restrict__ x,
                   const int32_t* __restrict__ dst_row, uint4* __restrict__ xp,
                   int max_rows, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int segv = nvec / nseg;
  for (int64_t u = warp_g; u < n_tok * nseg; u += nwarps) {
    const int64_t t = u / nseg;
    const int v_begin = static_cast<int>(u - t * nseg) * segv;
    const int v_end = v_begin + segv;
    // lane j < k holds the destination row of slot j
    const int32_t my_dst = checked_row(
        lane < k ? __ldg(dst_row + t * k + lane) : -1, max_rows, status);
    // a token with no kept slot (all dropped at capacity) is not read
    if (!__any_sync(0xffffffffu, my_dst >= 0)) continue;
    const uint4* src = x + t * nvec;
    // The step loop is warp-uniform (every lane runs every step, out-of-range
    // vectors masked) so that the full-mask shuffle below always has all 32
    // lanes: with a lane-strided bound, a segment shorter than 32 vectors, or
    // one whose length is 1-31 past a multiple of 128, would leave lanes out.
    for (int v0 = v_begin; v0 < v_end; v0 += 32 * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + lane + u * 32;
        if (v < v_end) buf[u] = ld_nc_v4(src + v);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_dst, j);
        if (r < 0) continue;
        uint4* dst = xp + static_cast<int64_t>(r) * nvec;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + lane + u * 32;
          if (v < v_end) st_v4(dst + v, buf[u]);
        }
      }
    }
  }
}

// SEG = false is the one-segment case with the segment arithmetic folded
// away (measured faster than the general loop run with nseg = 1).
template <typename T, bool SEG>
__global__ void __launch_bounds__(kRowWarps * 32)
    combine_kernel(int64_t n_tok, int k, int nvec, int nseg_arg,
                   const uint4* __restrict__ yp,
                   const int32_t* __restrict__ dst_row,
                   const float* __restrict__ gate, uint4* __restrict__ y,
                   int max_rows, int32_t* status) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int nseg = SEG ? nseg_arg : 1;
  const int segv = nvec / nseg;
  for (int64_t u = warp_g; u < n_tok * nseg; u += nwarps) {
    const int64_t t = u / nseg;
    const int v_begin = static_cast<int>(u - t * nseg) * segv;
    const int v_end = v_begin + segv;
    const int32_t my_dst = checked_row(
        lane < k ? __ldg(dst_row + t * k + lane) : -1, max_rows, status);
    // gate == nullptr: unit gates (the permute backward sums the rows)
    const float my_g =
        lane < k ? (gate != nullptr ? __ldg(gate + t * k + lane) : 1.0f)
                 : 0.0f;
    uint4* out = y + t * nvec;
    // warp-uniform step loop, as in permute_kernel: the shuffles need all
    // 32 lanes
    for (int v0 = v_begin; v0 < v_end; v0 += 32 * kUnroll) {
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
          const int v = v0 + lane + u * 32;
          if (v < v_end) buf[u] = ld_nc_v4(src + v);
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
        const int v = v0 + lane + u * 32;
        if (v < v_end) st_v4(out + v, Vec16<T>::from_f32(acc[u]));
      }
    }
  }
}

// k = KS <= 2: every slot's row vectors are loaded before any arithmetic,
// so a step costs one memory round trip instead of k; each vector is then
// reduced and stored on its own, so only its 8 (bf16) accumulators are live
// and the block fits 4 times per SM.  The fp32 operations and their
// order are combine_kernel's: y = fma(g1, x1, fma(g0, x0, 0)) (k = 2) or
// fma(g0, x0, 0) (k = 1), a dropped slot skipped.
template <typename T, bool SEG, int KS>
__global__ void __launch_bounds__(kRowWarps * 32, 4)
    combine2_kernel(int64_t n_tok, int nvec, int nseg_arg,
                    const uint4* __restrict__ yp,
                    const int32_t* __restrict__ dst_row,
                    const float* __restrict__ gate, uint4* __restrict__ y,
                    int max_rows, int32_t* status) {
  static_assert(KS == 1 || KS == 2, "one or two slots");
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int nseg = SEG ? nseg_arg : 1;
  const int segv = nvec / nseg;
  for (int64_t u = warp_g; u < n_tok * nseg; u += nwarps) {
    const int64_t t = u / nseg;
    const int v_begin = static_cast<int>(u - t * nseg) * segv;
    const int v_end = v_begin + segv;
    const int32_t my_dst = checked_row(
        lane < KS ? __ldg(dst_row + t * KS + lane) : -1, max_rows, status);
    const float my_g =
        lane < KS ? (gate != nullptr ? __ldg(gate + t * KS + lane) : 1.0f)
                  : 0.0f;
    const int32_t r0 = __shfl_sync(0xffffffffu, my_dst, 0);
    // lane 1 holds -1 when k = 1, so the second slot is skipped throughout
    const int32_t r1 = KS == 2 ? __shfl_sync(0xffffffffu, my_dst, 1) : -1;
    const float g0 = __shfl_sync(0xffffffffu, my_g, 0);
    const float g1 = KS == 2 ? __shfl_sync(0xffffffffu, my_g, 1) : 0.0f;
    const uint4* s0 = yp + static_cast<int64_t>(r0 < 0 ? 0 : r0) * nvec;
    const uint4* s1 = yp + static_cast<int64_t>(r1 < 0 ? 0 : r1) * nvec;
    uint4* out = y + t * nvec;
    for (int v0 = v_begin + lane; v0 < v_end; v0 += 32 * kUnroll) {
      uint4 b0[kUnroll], b1[kUnroll];
#pragma unroll
      for (int w = 0; w < kUnroll; ++w) {
        const int v = v0 + w * 32;
        const bool in = v < v_end;
        b0[w] = in && r0 >= 0 ? ld_nc_v4(s0 + v) : make_uint4(0u, 0u, 0u, 0u);
        b1[w] = in && r1 >= 0 ? ld_nc_v4(s1 + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int w = 0; w < kUnroll; ++w) {
        const int v = v0 + w * 32;
        if (v >= v_end) continue;
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = 0.0f;
        if (r0 >= 0) {
          float f[N];
          Vec16<T>::to_f32(b0[w], f);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] = fmaf(g0, f[i], acc[i]);
        }
        if (r1 >= 0) {
          float f[N];
          Vec16<T>::to_f32(b1[w], f);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] = fmaf(g1, f[i], acc[i]);
        }
        st_v4(out + v, Vec16<T>::from_f32(acc));
      }
    }
  }
}

// Segments per row: double while the warps would number fewer than 48 per
// SM and each segment keeps at least 128 vectors (one full step of 32 lanes
// x 4); a segment count always divides nvec.
static int row_segments(int64_t T, int nvec, int num_sms) {
  int nseg = 1;
  while (nseg < 4 && T * nseg < static_cast<int64_t>(num_sms) * 48 &&
         nvec % (2 * nseg) == 0 && nvec / (2 * nseg) >= 32 * kUnroll)
    nseg *= 2;
  return nseg;
}

static unsigned row_grid(int64_t units, int num_sms) {
  // enough resident warps to cover HBM latency: 8 blocks of 8 warps per SM
  const int64_t want = ceil_div(units, kRowWarps);
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<unsigned>(want < cap ? want : cap);
}

moe_status launch_permute(int T, int k, int D, int dtype, const void* x,
                          const int32_t* dst_row, void* xp, int max_rows,
                          int32_t* status, cudaStream_t stream, int num_sms) {
  if (T == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const int nseg = row_segments(T, nvec, num_sms);
  const unsigned grid = row_grid(static_cast<int64_t>(T) * nseg, num_sms);
  if (dtype == MOE_BF16)
    permute_kernel<__nv_bfloat16><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, nseg, static_cast<const uint4*>(x), dst_row,
        static_cast<uint4*>(xp), max_rows, status);
  else
    permute_kernel<float><<<grid, kRowWarps * 32, 0, stream>>>(
        T, k, nvec, nseg, static_cast<const uint4*>(x), dst_row,
        static_cast<uint4*>(xp), max_rows, status);
  return launch_status();
}

moe_status launch_combine(int T, int k, int D, int dtype, const void* yp,
                          const int32_t* dst_row, const float* gate, void* y,
                          int max_rows, int32_t* status, cudaStream_t stream,
                          int num_sms) {
  if (T == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  // with more than 4 slots a token's gather already has enough independent
  // loads; splitting its row measured slower (k = 8)
  const int nseg = k <= 4 ? row_segments(T, nvec, num_sms) : 1;
  const unsigned grid = row_grid(static_cast<int64_t>(T) * nseg, num_sms);
  const uint4* src = static_cast<const uint4*>(yp);
  uint4* dst = static_cast<uint4*>(y);
  if (k == 2 && dtype == MOE_BF16) {
    if (nseg > 1)
      combine2_kernel<__nv_bfloat16, true, 2><<<grid, kRowWarps * 32, 0, stream>>>(
          T, nvec, nseg, src, dst_row, gate, dst, max_rows, status);
    else
      combine2_kernel<__nv_bfloat16, false, 2><<<grid, kRowWarps * 32, 0, stream>>>(
          T, nvec, 1, src, dst_row, gate, dst, max_rows, status);
    return launch_status();
  }
  if (k == 1 && dtype == MOE_BF16) {
    if (nseg > 1)
      combine2_kernel<__nv_bfloat16, true, 1><<<grid, kRowWarps * 32, 0, stream>>>(
          T, nvec, nseg, src, dst_row, gate, dst, max_rows, status);
    else
      combine2_kernel<__nv_bfloat16, false, 1><<<grid, kRowWarps * 32, 0, stream>>>(
          T, nvec, 1, src, dst_row, gate, dst, max_rows, status);
    return launch_status();
  }
  if (dtype == MOE_BF16) {
    if (nseg > 1)
      combine_kernel<__nv_bfloat16, true><<<grid, kRowWarps * 32, 0, stream>>>(
          T, k, nvec, nseg, src, dst_row, gate, dst, max_rows, status);
    else
      combine_kernel<__nv_bfloat16, false><<<grid, kRowWarps * 32, 0, stream>>>(
          T, k, nvec, 1, src, dst_row, gate, dst, max_rows, status);
  } else {
    if (nseg > 1)
      combine_kernel<float, true><<<grid, kRowWarps * 32, 0, stream>>>(
          T, k, nvec, nseg, src, dst_row, gate, dst, max_rows, status);
    else
      combine_kernel<float, false><<<grid, kRowWarps * 32, 0, stream>>>(
          T, k, nvec, 1, src, dst_row, gate, dst, max_rows, status);
  }
  return launch_status();
}

}  // namespace moe
