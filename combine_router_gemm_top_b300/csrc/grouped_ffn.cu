// moe_grouped_ffn: per-expert SwiGLU over ragged, expert-contiguous row
// segments ("Expert Parallelism in LLMs", The Execution Pipeline, step 4
// "Local Expert Computation": the tokens of one expert packed into one
// GEMM; Modern Dropless Dynamic Dispatch: ragged grouped GEMM on exact
// per-expert counts, no padding).
//
// bf16: two persistent tcgen05 launches over a device-side tile list built
// from expert_offsets (no host synchronisation):
//   up    H[r, n:n+128]  = SiLU(Xp W1^T) * (Xp W3^T) for a 128-row block of
//         one expert; B tile = 128 W1 rows stacked on the matching 128 W3
//         rows, so gate and up land in one 128 x 256 TMEM accumulator and
//         the GLU is applied in the epilogue (H rounded to bf16).
//   down  Yp[r, n:n+256] = H W2^T.
// Tiles run m-block-fastest inside (expert, n-block), so the CTAs working
// at the same time share the weight tile through L2.
// fp32: plain FMA kernels, one thread per output element.
#include "common.cuh"
#include "internal.h"
#include "umma_ffn.cuh"
#include "umma_ffn_pair.cuh"
#include "umma_gemm.cuh"

namespace moe {

// ----------------------------------------------------------- fp32 path
__device__ __forceinline__ int find_expert(const int32_t* off, int E, int row) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One warp per row and kFpw consecutive outputs: the lanes stride over the
// dot products' length, so every load of x, H and the weight rows is
// coalesced and each x (H) element loaded serves kFpw outputs; a shuffle tree
// adds the lanes' parts in a fixed order.
constexpr int kFpw = 4;

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void ffn_up_f32_kernel(int E, int D, int F, int max_rows,
                                  const float* __restrict__ xp,
                                  const int32_t* __restrict__ off,
                                  const float* __restrict__ w13,
                                  float* __restrict__ h) {
  const int64_t i =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int n_rows = min(__ldg(off + E), max_rows);
  const int fg = (F + kFpw - 1) / kFpw;   // feature groups per row
  if (i >= static_cast<int64_t>(n_rows) * fg) return;   // warp-uniform
  const int row = static_cast<int>(i / fg);
  const int f0 = static_cast<int>(i - static_cast<int64_t>(row) * fg) * kFpw;
  const int e = find_expert(off, E, row);
  const float* x = xp + static_cast<int64_t>(row) * D;
  const float* w1 = w13 + (static_cast<int64_t>(e) * 2 * F + f0) * D;
  const float* w3 = w1 + static_cast<int64_t>(F) * D;
  const int nf = min(kFpw, F - f0);
  float g[kFpw], u[kFpw];
#pragma unroll
  for (int j = 0; j < kFpw; ++j) g[j] = u[j] = 0.0f;
  for (int d = lane; d < D; d += 32) {
    const float xv = __ldg(x + d);
#pragma unroll
    for (int j = 0; j < kFpw; ++j) {
      if (j < nf) {
        g[j] = fmaf(xv, __ldg(w1 + static_cast<int64_t>(j) * D + d), g[j]);
        u[j] = fmaf(xv, __ldg(w3 + static_cast<int64_t>(j) * D + d), u[j]);
      }
    }
  }
  float out = 0.0f;
#pragma unroll
  for (int j = 0; j < kFpw; ++j) {
    const float gs = warp_sum_f32(g[j]);
    const float us = warp_sum_f32(u[j]);
    if (lane == j) out = gs / (1.0f + expf(-gs)) * us;
  }
  if (lane < nf) h[static_cast<int64_t>(row) * F + f0 + lane] = out;
}

__global__ void ffn_down_f32_kernel(int E, int D, int F, int max_rows,
                                    const float* __restrict__ h,
                                    const int32_t* __restrict__ off,
                                    const float* __restrict__ w2,
                                    float* __restrict__ yp) {
  const int64_t i =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int n_rows = min(__ldg(off + E), max_rows);
  const int dg = (D + kFpw - 1) / kFpw;   // output groups per row
  if (i >= static_cast<int64_t>(n_rows) * dg) return;   // warp-uniform
  const int row = static_cast<int>(i / dg);
  const int d0 = static_cast<int>(i - static_cast<int64_t>(row) * dg) * kFpw;
  const int e = find_expert(off, E, row);
  const float* hr = h + static_cast<int64_t>(row) * F;
  const float* w = w2 + (static_cast<int64_t>(e) * D + d0) * F;
  const int nd = min(kFpw, D - d0);
  float acc[kFpw];
#pragma unroll
  for (int j = 0; j < kFpw; ++j) acc[j] = 0.0f;
  for (int f = lane; f < F; f += 32) {
    const float hv = __ldg(hr + f);
#pragma unroll
    for (int j = 0; j < kFpw; ++j)
      if (j < nd)
        acc[j] = fmaf(hv, __ldg(w + static_cast<int64_t>(j) * F + f), acc[j]);
  }
  float out = 0.0f;
#pragma unroll
  for (int j = 0; j < kFpw; ++j) {
    const float s = warp_sum_f32(acc[j]);
    if (lane == j) out = s;
  }
  if (lane < nd) yp[static_cast<int64_t>(row) * D + d0 + lane] = out;
}

// The same two projections for one row in one block: its H row stays in
// shared memory (F fp32 values) between them, and each output is formed in
// the same order as by the two kernels above, so the results are the same
// bits.  One launch, and H never goes to HBM.
constexpr int kRowFfnMaxF = 12288;   // 48 KB of H per block

__global__ void __launch_bounds__(256)
    ffn_row_f32_kernel(int E, int D, int F, int max_rows,
                       const float* __restrict__ xp,
                       const int32_t* __restrict__ off,
                       const float* __restrict__ w13,
                       const float* __restrict__ w2,
                       float* __restrict__ yp) {
  extern __shared__ float hs[];   // [F]
  const int row = blockIdx.x;
  const int n_rows = min(__ldg(off + E), max_rows);
  if (row >= n_rows) return;   // block-uniform
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int e = find_expert(off, E, row);
  const float* x = xp + static_cast<int64_t>(row) * D;
  for (int f0 = kFpw * warp; f0 < F; f0 += kFpw * nw) {
    const float* w1 = w13 + (static_cast<int64_t>(e) * 2 * F + f0) * D;
    const float* w3 = w1 + static_cast<int64_t>(F) * D;
    const int nf = min(kFpw, F - f0);
    float g[kFpw], u[kFpw];
#pragma unroll
    for (int j = 0; j < kFpw; ++j) g[j] = u[j] = 0.0f;
    for (int d = lane; d < D; d += 32) {
      const float xv = __ldg(x + d);
#pragma unroll
      for (int j = 0; j < kFpw; ++j) {
        if (j < nf) {
          g[j] = fmaf(xv, __ldg(w1 + static_cast<int64_t>(j) * D + d), g[j]);
          u[j] = fmaf(xv, __ldg(w3 + static_cast<int64_t>(j) * D + d), u[j]);
        }
      }
    }
    float out = 0.0f;
#pragma unroll
    for (int j = 0; j < kFpw; ++j) {
      const float gs = warp_sum_f32(g[j]);
      const float us = warp_sum_f32(u[j]);
      if (lane == j) out = gs / (1.0f + expf(-gs)) * us;
    }
    if (lane < nf) hs[f0 + lane] = out;
  }
  __syncthreads();
  for (int d0 = kFpw * warp; d0 < D; d0 += kFpw * nw) {
    const float* w = w2 + (static_cast<int64_t>(e) * D + d0) * F;
    const int nd = min(kFpw, D - d0);
    float acc[kFpw];
#pragma unroll
    for (int j = 0; j < kFpw; ++j) acc[j] = 0.0f;
    for (int f = lane; f < F; f += 32) {
      const float hv = hs[f];
#pragma unroll
      for (int j = 0; j < kFpw; ++j)
        if (j < nd)
          acc[j] = fmaf(hv, __ldg(w + static_cast<int64_t>(j) * F + f), acc[j]);
    }
    float out = 0.0f;
#pragma unroll
    for (int j = 0; j < kFpw; ++j) {
      const float s = warp_sum_f32(acc[j]);
      if (lane == j) out = s;
    }
    if (lane < nd) yp[static_cast<int64_t>(row) * D + d0 + lane] = out;
  }
}

// ----------------------------------------------------------- host
// Workspace: H [max_rows, F], then (bf16) one ready counter per row block of
// the fused launch (at most ceil(max_rows / 128) + E blocks) and the SM-pair
// launch's tile ticket.
static size_t ffn_h_bytes(int F, int max_rows, int dtype) {
  return (static_cast<size_t>(max_rows) * F * dtype_bytes(dtype) + 255) &
         ~size_t(255);
}
static int ffn_ready_cap(int E, int max_rows) {
  return static_cast<int>(ceil_div(max_rows, kBM)) + E;
}

size_t ffn_ws_bytes(int E, int D, int F, int max_rows, int dtype) {
  (void)D;
  if (dtype != MOE_BF16)
    return static_cast<size_t>(max_rows) * F * dtype_bytes(dtype);
  return ffn_h_bytes(F, max_rows, dtype) +
         static_cast<size_t>(ffn_ready_cap(E, max_rows) + 1) * sizeof(uint32_t);
}

int ffn_variant(int E, int F, int max_rows, int dtype) {
  if (dtype == MOE_F32) return F <= kRowFfnMaxF ? 1 : 4;
  // SM pairs when the experts average at least 1.5 pair row blocks (256
  // rows): below that the 256-row blocks waste more rows than the pairs
  // save
  return F % 256 == 0 && E <= kPairMaxGroups &&
                 static_cast<int64_t>(max_rows) >= 384LL * E
             ? 3
             : 2;
}

// SM pairs (umma_ffn_pair.cuh): persistent 2-CTA clusters, at most as many
// as fit at once (more would only find the tile ticket used up).  Tiles are
// claimed in order, so no cluster waits on one that is not running and the
// launch needs no co-residency guarantee.
static moe_status launch_ffn_pair(int E, int D, int F, int max_rows,
                                  const void* xp, const int32_t* offsets,
                                  const void* w13, const void* w2, void* yp,
                                  void* h, uint32_t* ready, int ready_cap,
                                  int max_ctas, int32_t* status,
                                  cudaStream_t stream, int num_sms) {
  CUtensorMap tm_xp, tm_w13, tm_h, tm_w2, tm_xp_t, tm_h_t;
  if (!make_tmap_bf16_2d(&tm_xp, xp, D, max_rows, 128) ||
      !make_tmap_bf16_2d(&tm_w13, w13, D, static_cast<int64_t>(E) * 2 * F, 128) ||
      !make_tmap_bf16_2d(&tm_h, h, F, max_rows, 128) ||
      !make_tmap_bf16_2d(&tm_w2, w2, F, static_cast<int64_t>(E) * D, 128) ||
      !make_tmap_bf16_2d(&tm_xp_t, xp, D, max_rows, kPairSwapMax / 2) ||
      !make_tmap_bf16_2d(&tm_h_t, h, F, max_rows, kPairSwapMax / 2))
    return MOE_ERR_CUDA;
  PairFfnArgs a{};
  a.E = E;
  a.D = D;
  a.F = F;
  a.kb_up = D / kBK;
  a.kb_dn = F / kBK;
  a.n_up = F / 128;
  a.S = F / 256;
  a.n_dn = static_cast<int>(ceil_div(D, 256));
  a.offsets = offsets;
  a.max_rows = max_rows;
  a.h = static_cast<__nv_bfloat16*>(h);
  a.yp = static_cast<__nv_bfloat16*>(yp);
  a.ready = ready;
  a.ready_cap = ready_cap;
  a.ticket = ready + ready_cap;
  a.status = status;
  a.wait_limit_ns = kWaitLimitNs;
  static std::atomic<uint64_t> attr_done{0};
  if (!set_smem_limit_once(reinterpret_cast<const void*>(umma_ffn_pair_kernel),
                           227 * 1024, &attr_done))
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = umma_ffn_pair_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, umma_ffn_pair_kernel, &cfg) !=
          cudaSuccess ||
      clusters < 1) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  int want = max_ctas > 0 && max_ctas < num_sms ? max_ctas / 2 : num_sms / 2;
  if (want < 1) want = 1;
  cfg.gridDim =
      dim3(static_cast<unsigned>(2 * (want < clusters ? want : clusters)));
  if (cudaLaunchKernelEx(&cfg, umma_ffn_pair_kernel, tm_xp, tm_w13, tm_h,
                         tm_w2, tm_xp_t, tm_h_t, a) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}


moe_status launch_grouped_ffn(int E, int D, int F, int max_rows, int dtype,
                              const void* xp, const int32_t* offsets,
                              const void* w13, const void* w2, void* yp,
                              void* ws, int max_ctas, int32_t* status,
                              cudaStream_t stream, int num_sms) {
  if (max_rows == 0) return MOE_OK;
  if (dtype == MOE_F32 && ffn_variant(E, F, max_rows, dtype) == 1) {
    ffn_row_f32_kernel<<<static_cast<unsigned>(max_rows), 256,
                         static_cast<size_t>(F) * sizeof(float), stream>>>(
        E, D, F, max_rows, static_cast<const float*>(xp), offsets,
        static_cast<const float*>(w13), static_cast<const float*>(w2),
        static_cast<float*>(yp));
    return launch_status();
  }
  if (dtype == MOE_F32) {
    float* h = static_cast<float*>(ws);
    // one warp per row and kFpw outputs, 8 warps a block
    const int64_t n1 = static_cast<int64_t>(max_rows) * ceil_div(F, kFpw);
    const int64_t n2 = static_cast<int64_t>(max_rows) * ceil_div(D, kFpw);
    if (ceil_div(n1, 8) > INT32_MAX || ceil_div(n2, 8) > INT32_MAX)
      return MOE_ERR_UNSUPPORTED;
    ffn_up_f32_kernel<<<static_cast<unsigned>(ceil_div(n1, 8)), 256, 0,
                        stream>>>(E, D, F, max_rows,
                                  static_cast<const float*>(xp), offsets,
                                  static_cast<const float*>(w13), h);
    ffn_down_f32_kernel<<<static_cast<unsigned>(ceil_div(n2, 8)), 256, 0,
                          stream>>>(E, D, F, max_rows, h, offsets,
                                    static_cast<const float*>(w2),
                                    static_cast<float*>(yp));
    return launch_status();
  }
  void* h = ws;
  CUtensorMap tm_xp, tm_w13, tm_h, tm_w2;
  if (!make_tmap_bf16_2d(&tm_xp, xp, D, max_rows, kBM) ||
      !make_tmap_bf16_2d(&tm_w13, w13, D, static_cast<int64_t>(E) * 2 * F, 128) ||
      !make_tmap_bf16_2d(&tm_h, h, F, max_rows, kBM) ||
      !make_tmap_bf16_2d(&tm_w2, w2, F, static_cast<int64_t>(E) * D, 256))
    return MOE_ERR_CUDA;

  GemmArgs up{};
  up.M = max_rows;
  up.k_blocks = D / kBK;
  up.BN = 256;
  up.stages = 4;
  up.tmem_cols = 512;
  up.groups = E;
  up.n_tiles = F / 128;
  up.F = F;
  up.b_rows_per_group = 2 * F;
  up.offsets = offsets;
  up.out = h;
  up.out_ld = F;
  up.out_cols = F;
  up.status = status;
  up.wait_limit_ns = kWaitLimitNs;

  GemmArgs dn = up;
  dn.k_blocks = F / kBK;
  dn.n_tiles = static_cast<int>(ceil_div(D, 256));
  dn.F = 0;
  dn.b_rows_per_group = D;
  dn.out = yp;
  dn.out_ld = D;
  dn.out_cols = D;

  // up and down projection in one persistent launch (umma_ffn.cuh)
  FfnArgs f{};
  f.up = up;
  f.dn = dn;
  f.ready = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) +
                                        ffn_h_bytes(F, max_rows, dtype));
  f.ready_cap = ffn_ready_cap(E, max_rows);
  if (cudaMemsetAsync(f.ready, 0, static_cast<size_t>(f.ready_cap + 1) *
                                      sizeof(uint32_t),
                      stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ffn_variant(E, F, max_rows, dtype) == 3)
    return launch_ffn_pair(E, D, F, max_rows, xp, offsets, w13, w2, yp, h,
                           f.ready, f.ready_cap, max_ctas, status, stream,
                           num_sms);
  static std::atomic<uint64_t> attr_done{0};
  if (!set_smem_limit_once(reinterpret_cast<const void*>(umma_ffn_kernel),
                           227 * 1024, &attr_done))
    return MOE_ERR_CUDA;
  const size_t smem = umma_gemm_smem_bytes(up.BN, up.stages);
  // Down tiles wait for up tiles that other CTAs own, so every CTA of the
  // grid must be resident at once: a cooperative launch guarantees that (or
  // fails to launch), whatever else runs on the device.  One CTA per SM at
  // most, fewer when the caller asks.
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, umma_ffn_kernel, kGemmThreads, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  const int grid = max_ctas > 0 && max_ctas < num_sms ? max_ctas : num_sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, umma_ffn_kernel, tm_xp, tm_w13, tm_h, tm_w2,
                         f) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// ----------------------------------------------------------- self-test
// Waits on a barrier that nothing arrives on; the bounded wait must expire,
// raise the abort flag and report MOE_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    if (!ok && abort_flag) set_status(status, MOE_ERR_TIMEOUT);
  }
}

moe_status launch_selftest_wait(int32_t* status, uint64_t limit_ns,
                                cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return launch_status();
}

}  // namespace moe

namespace moe {

// ----------------------------------------------------------- backward
// Workspace of the backward: dH [rows, F], dGU [rows, 2F], H [rows, F]
// (bf16 each).
size_t ffn_bwd_ws_bytes(int F, int max_rows, int dtype) {
  return static_cast<size_t>(max_rows) * F * 4 * dtype_bytes(dtype);
}

// fp32 backward on the CUDA cores: one thread per output element, fp32
// accumulation in index order (the reference-precision path).
__global__ void ffn_bwd_dh_f32_kernel(int E, int D, int F, int max_rows,
                                      const int32_t* __restrict__ off,
                                      const float* __restrict__ dyp,
                                      const float* __restrict__ w2,
                                      float* __restrict__ dh) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int n_rows = min(__ldg(off + E), max_rows);
  if (i >= static_cast<int64_t>(n_rows) * F) return;
  const int row = static_cast<int>(i / F);
  const int f = static_cast<int>(i - static_cast<int64_t>(row) * F);
  const int e = find_expert(off, E, row);
  const float* g = dyp + static_cast<int64_t>(row) * D;
  const float* w = w2 + static_cast<int64_t>(e) * D * F + f;
  float acc = 0.0f;
  for (int d = 0; d < D; ++d) acc = fmaf(g[d], w[static_cast<int64_t>(d) * F], acc);
  dh[i] = acc;
}

// recomputes gate g and up u, then dG = dH u SiLU'(g), dU = dH SiLU(g) into
// dgu [rows, 2F] (W13's row order) and H = SiLU(g) u
__global__ void ffn_bwd_act_f32_kernel(int E, int D, int F, int max_rows,
                                       const int32_t* __restrict__ off,
                                       const float* __restrict__ xp,
                                       const float* __restrict__ w13,
                                       const float* __restrict__ dh,
                                       float* __restrict__ dgu,
                                       float* __restrict__ h) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int n_rows = min(__ldg(off + E), max_rows);
  if (i >= static_cast<int64_t>(n_rows) * F) return;
  const int row = static_cast<int>(i / F);
  const int f = static_cast<int>(i - static_cast<int64_t>(row) * F);
  const int e = find_expert(off, E, row);
  const float* x = xp + static_cast<int64_t>(row) * D;
  const float* w1 = w13 + (static_cast<int64_t>(e) * 2 * F + f) * D;
  const float* w3 = w1 + static_cast<int64_t>(F) * D;
  float g = 0.0f, u = 0.0f;
  for (int d = 0; d < D; ++d) {
    g = fmaf(x[d], w1[d], g);
    u = fmaf(x[d], w3[d], u);
  }
  const float s = 1.0f / (1.0f + expf(-g));
  const float d = dh[i];
  float* o = dgu + static_cast<int64_t>(row) * 2 * F;
  o[f] = d * u * s * (1.0f + g * (1.0f - s));
  o[F + f] = d * g * s;
  h[i] = g * s * u;
}

__global__ void ffn_bwd_dx_f32_kernel(int E, int D, int F, int max_rows,
                                      const int32_t* __restrict__ off,
                                      const float* __restrict__ dgu,
                                      const float* __restrict__ w13,
                                      float* __restrict__ dxp) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int n_rows = min(__ldg(off + E), max_rows);
  if (i >= static_cast<int64_t>(n_rows) * D) return;
  const int row = static_cast<int>(i / D);
  const int d = static_cast<int>(i - static_cast<int64_t>(row) * D);
  const int e = find_expert(off, E, row);
  const float* g = dgu + static_cast<int64_t>(row) * 2 * F;
  const float* w = w13 + static_cast<int64_t>(e) * 2 * F * D + d;
  float acc = 0.0f;
  for (int f = 0; f < 2 * F; ++f)
    acc = fmaf(g[f], w[static_cast<int64_t>(f) * D], acc);
  dxp[i] = acc;
}

// out[e, m, n] = sum over the rows r of expert e of a[r, m] * b[r, n]
__global__ void ffn_bwd_wgrad_f32_kernel(int E, int M, int N, int max_rows,
                                         const int32_t* __restrict__ off,
                                         const float* __restrict__ a, int lda,
                                         const float* __restrict__ b, int ldb,
                                         float* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(E) * M * N) return;
  const int e = static_cast<int>(i / (static_cast<int64_t>(M) * N));
  const int64_t mn = i - static_cast<int64_t>(e) * M * N;
  const int m = static_cast<int>(mn / N);
  const int n = static_cast<int>(mn - static_cast<int64_t>(m) * N);
  const int r0 = min(__ldg(off + e), max_rows);
  const int r1 = min(__ldg(off + e + 1), max_rows);
  float acc = 0.0f;
  for (int r = r0; r < r1; ++r)
    acc = fmaf(a[static_cast<int64_t>(r) * lda + m],
               b[static_cast<int64_t>(r) * ldb + n], acc);
  out[i] = acc;
}

moe_status launch_grouped_ffn_backward_f32(int E, int D, int F, int max_rows,
                                           const float* xp, const float* dyp,
                                           const int32_t* off,
                                           const float* w13, const float* w2,
                                           float* dxp, float* dw13, float* dw2,
                                           void* ws, cudaStream_t stream) {
  float* dh = static_cast<float*>(ws);
  float* dgu = dh + static_cast<size_t>(max_rows) * F;
  float* h = dgu + static_cast<size_t>(max_rows) * 2 * F;
  auto grid = [](int64_t n) {
    return static_cast<unsigned>(ceil_div(n > 0 ? n : 1, 256));
  };
  const int64_t rf = static_cast<int64_t>(max_rows) * F;
  const int64_t rd = static_cast<int64_t>(max_rows) * D;
  ffn_bwd_dh_f32_kernel<<<grid(rf), 256, 0, stream>>>(E, D, F, max_rows, off,
                                                      dyp, w2, dh);
  ffn_bwd_act_f32_kernel<<<grid(rf), 256, 0, stream>>>(E, D, F, max_rows, off,
                                                       xp, w13, dh, dgu, h);
  ffn_bwd_dx_f32_kernel<<<grid(rd), 256, 0, stream>>>(E, D, F, max_rows, off,
                                                      dgu, w13, dxp);
  const int64_t n2 = static_cast<int64_t>(E) * D * F;
  ffn_bwd_wgrad_f32_kernel<<<grid(n2), 256, 0, stream>>>(
      E, D, F, max_rows, off, dyp, D, h, F, dw2);
  const int64_t n13 = static_cast<int64_t>(E) * 2 * F * D;
  ffn_bwd_wgrad_f32_kernel<<<grid(n13), 256, 0, stream>>>(
      E, 2 * F, D, max_rows, off, dgu, 2 * F, xp, D, dw13);
  return launch_status();
}

moe_status launch_grouped_ffn_backward(int E, int D, int F, int max_rows,
                                       const void* xp, const void* dyp,
                                       const int32_t* offsets,
                                       const void* w13, const void* w2,
                                       void* dxp, float* dw13, float* dw2,
                                       void* ws, int32_t* status,
                                       cudaStream_t stream, int num_sms) {
  if (max_rows == 0) return MOE_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t rf = static_cast<size_t>(max_rows) * F * 2;
  void* dh = w;
  void* dgu = w + rf;
  void* h = w + 3 * rf;
  const int64_t EF2 = static_cast<int64_t>(E) * 2 * F;
  const int64_t ED = static_cast<int64_t>(E) * D;
  CUtensorMap t_dyp, t_w2mn, t_xp, t_w13, t_dgu, t_w13mn, t_dyp_mn, t_h_mn,
      t_dgu_mn, t_xp_mn;
  if (!make_tmap_bf16_2d(&t_dyp, dyp, D, max_rows, kBM) ||
      !make_tmap_bf16_2d(&t_w2mn, w2, F, ED, 64) ||
      !make_tmap_bf16_2d(&t_xp, xp, D, max_rows, kBM) ||
      !make_tmap_bf16_2d(&t_w13, w13, D, EF2, 128) ||
      !make_tmap_bf16_2d(&t_dgu, dgu, 2 * F, max_rows, kBM) ||
      !make_tmap_bf16_2d(&t_w13mn, w13, D, EF2, 64) ||
      !make_tmap_bf16_2d(&t_dyp_mn, dyp, D, max_rows, 64) ||
      !make_tmap_bf16_2d(&t_h_mn, h, F, max_rows, 64) ||
      !make_tmap_bf16_2d(&t_dgu_mn, dgu, 2 * F, max_rows, 64) ||
      !make_tmap_bf16_2d(&t_xp_mn, xp, D, max_rows, 64))
    return MOE_ERR_CUDA;

  GemmArgs base{};
  base.M = max_rows;
  base.BN = 256;
  base.stages = 4;
  base.tmem_cols = 512;
  base.groups = E;
  base.F = F;
  base.offsets = offsets;
  base.status = status;
  base.wait_limit_ns = kWaitLimitNs;

  // dH = dYp . W2_e   (B = W2 [D, F] read MN-major)
  GemmArgs g = base;
  g.k_blocks = D / kBK;
  g.n_tiles = static_cast<int>(ceil_div(F, 256));
  g.b_rows_per_group = D;
  g.out = dh;
  g.out_ld = F;
  g.out_cols = F;
  moe_status s = launch_umma<kDH>(t_dyp, t_w2mn, g, stream, num_sms);
  if (s != MOE_OK) return s;

  // recompute gate/up, then dG, dU (into dGU) and H
  g = base;
  g.k_blocks = D / kBK;
  g.n_tiles = F / 128;
  g.b_rows_per_group = 2 * F;
  g.aux_in = dh;
  g.out = dgu;
  g.out2 = h;
  g.out_ld = F;
  g.out_cols = F;
  s = launch_umma<kUpBwd>(t_xp, t_w13, g, stream, num_sms);
  if (s != MOE_OK) return s;

  // dXp = dGU . W13_e   (B = W13 [2F, D] read MN-major)
  g = base;
  g.k_blocks = 2 * F / kBK;
  g.n_tiles = static_cast<int>(ceil_div(D, 256));
  g.b_rows_per_group = 2 * F;
  g.out = dxp;
  g.out_ld = D;
  g.out_cols = D;
  s = launch_umma<kDX>(t_dgu, t_w13mn, g, stream, num_sms);
  if (s != MOE_OK) return s;

  // dW2_e = dYp_e^T . H_e   [D, F] per expert, fp32 (3 stages leave room
  // for the epilogue's staging tiles)
  g = base;
  g.stages = 3;
  g.m_total = D;
  g.m_tiles = D / kBM;
  g.n_tiles = static_cast<int>(ceil_div(F, 256));
  g.M = static_cast<int32_t>(ED);
  g.n_fast = D > F;   // keep the narrower operand (H or dYp) in L2
  g.out = dw2;
  g.out_ld = F;
  g.out_cols = F;
  s = launch_umma<kWG2>(t_dyp_mn, t_h_mn, g, stream, num_sms);
  if (s != MOE_OK) return s;

  // dW13_e = dGU_e^T . Xp_e   [2F, D] per expert, fp32
  g = base;
  g.stages = 3;
  g.m_total = 2 * F;
  g.m_tiles = 2 * F / kBM;
  g.n_tiles = static_cast<int>(ceil_div(D, 256));
  g.M = static_cast<int32_t>(EF2);
  g.n_fast = 2 * F > D;   // keep the narrower operand (Xp or [dG|dU]) in L2
  g.out = dw13;
  g.out_ld = D;
  g.out_cols = D;
  return launch_umma<kWG13>(t_dgu_mn, t_xp_mn, g, stream, num_sms);
}

}  // namespace moe
