// Router statistics of one routing decision ("Expert Parallelism in LLMs",
// Static Capacity Factors and Token Dropping: the auxiliary load-balancing
// loss L_aux = alpha * E * sum_i f_i * P_i, f_i the fraction of routed
// pairs on expert i, P_i the mean router probability of expert i) and the
// auxiliary-loss-free bias step (same page, Modern Dropless Dynamic
// Dispatch: bias terms on the routing scores adjusted to keep the load
// balanced).
//
// Two deterministic launches: per-block partial sums (fp64 probability
// sums, int32 routed counts) over a fixed token order, then one block of 32
// warps that adds the partials in a fixed order and forms f, P and L_aux.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStatsWarps = 8;

__device__ __forceinline__ float stats_warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float stats_warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// One warp per token (grid-stride); lane l holds experts l + 32 i.
template <int NI>
__global__ void __launch_bounds__(kStatsWarps * 32)
    router_stats_partial_kernel(int T, int E, int k, int score,
                                const float* __restrict__ logits,
                                const int32_t* __restrict__ topk_idx,
                                double* __restrict__ part_p,
                                int32_t* __restrict__ part_cnt,
                                int32_t* status) {
  __shared__ double s_p[kStatsWarps][NI * 32];
  __shared__ int32_t s_cnt[NI * 32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < NI * 32; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();

  double acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0.0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kStatsWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kStatsWarps + warp;
       t < T; t += stride) {
    float l[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      l[i] = e < E ? logits[t * E + e] : 0.0f;
    }
    float p[NI];
    if (score == MOE_SCORE_SIGMOID_BIAS) {
      float z = 0.0f;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        p[i] = lane + 32 * i < E ? 1.0f / (1.0f + expf(-l[i])) : 0.0f;
        z += p[i];
      }
      z = stats_warp_sum(z);
#pragma unroll
      for (int i = 0; i < NI; ++i) p[i] = p[i] / z;
    } else {
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (lane + 32 * i < E) m = fmaxf(m, l[i]);
      m = stats_warp_max(m);
      float z = 0.0f;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        p[i] = lane + 32 * i < E ? expf(l[i] - m) : 0.0f;
        z += p[i];
      }
      z = stats_warp_sum(z);
#pragma unroll
      for (int i = 0; i < NI; ++i) p[i] = p[i] / z;
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) acc[i] += static_cast<double>(p[i]);
    if (lane < k) {
      const int e = topk_idx[t * k + lane];
      if (e >= 0 && e < E)
        atomicAdd(&s_cnt[e], 1);
      else
        set_status(status, MOE_ERR_INDEX);
    }
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) s_p[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double s = 0.0;
    for (int w = 0; w < kStatsWarps; ++w) s += s_p[w][e];
    part_p[static_cast<int64_t>(blockIdx.x) * E + e] = s;
    part_cnt[static_cast<int64_t>(blockIdx.x) * E + e] = s_cnt[e];
  }
}

// One block of 32 warps: warp w sums the partials of experts w, w+32, ...
// (lane-strided over blocks, then a fixed xor tree), and the block adds
// f_i * P_i over experts in a fixed order.  Deterministic.
constexpr int kFinalWarps = 32;

__global__ void __launch_bounds__(kFinalWarps * 32)
    router_stats_final_kernel(int T, int E, int k, int blocks, float alpha,
                              const double* __restrict__ part_p,
                              const int32_t* __restrict__ part_cnt,
                              float* __restrict__ f, float* __restrict__ P,
                              int32_t* __restrict__ counts_routed,
                              float* __restrict__ aux_loss) {
  __shared__ double s_fp[kFinalWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const double pairs = static_cast<double>(T) * k;
  double local = 0.0;
  for (int e = warp; e < E; e += kFinalWarps) {
    double sp = 0.0;
    long long c = 0;
    for (int b = lane; b < blocks; b += 32) {
      sp += part_p[static_cast<int64_t>(b) * E + e];
      c += part_cnt[static_cast<int64_t>(b) * E + e];
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      sp += __shfl_xor_sync(0xffffffffu, sp, d);
      c += __shfl_xor_sync(0xffffffffu, c, d);
    }
    const double fe = pairs > 0 ? static_cast<double>(c) / pairs : 0.0;
    const double pe = T > 0 ? sp / static_cast<double>(T) : 0.0;
    if (lane == 0) {
      f[e] = static_cast<float>(fe);
      P[e] = static_cast<float>(pe);
      if (counts_routed != nullptr) counts_routed[e] = static_cast<int32_t>(c);
    }
    local += fe * pe;
  }
  if (lane == 0) s_fp[warp] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kFinalWarps; ++w) s += s_fp[w];
    aux_loss[0] = static_cast<float>(static_cast<double>(alpha) * E * s);
  }
}

int router_stats_blocks(int T) {
  const int64_t want = ceil_div(T, kStatsWarps);
  return static_cast<int>(want < kNumSMs ? (want > 0 ? want : 1) : kNumSMs);
}

size_t router_stats_ws_bytes(int T, int E) {
  const size_t b = static_cast<size_t>(router_stats_blocks(T));
  return b * E * (sizeof(double) + sizeof(int32_t)) + 256;
}

moe_status launch_router_stats(int T, int E, int k, int score,
                               const float* logits, const int32_t* topk_idx,
                               float alpha, float* f, float* P,
                               int32_t* counts_routed, float* aux_loss,
                               void* ws, int32_t* status,
                               cudaStream_t stream) {
  const int blocks = router_stats_blocks(T);
  double* part_p = static_cast<double*>(ws);
  int32_t* part_cnt = reinterpret_cast<int32_t*>(
      static_cast<uint8_t*>(ws) + static_cast<size_t>(blocks) * E * sizeof(double));
  const int ni = static_cast<int>(ceil_div(E, 32));
  const dim3 grid(static_cast<unsigned>(blocks)), block(kStatsWarps * 32);
  if (ni <= 1)
    router_stats_partial_kernel<1><<<grid, block, 0, stream>>>(
        T, E, k, score, logits, topk_idx, part_p, part_cnt, status);
  else if (ni <= 2)
    router_stats_partial_kernel<2><<<grid, block, 0, stream>>>(
        T, E, k, score, logits, topk_idx, part_p, part_cnt, status);
  else if (ni <= 4)
    router_stats_partial_kernel<4><<<grid, block, 0, stream>>>(
        T, E, k, score, logits, topk_idx, part_p, part_cnt, status);
  else
    router_stats_partial_kernel<8><<<grid, block, 0, stream>>>(
        T, E, k, score, logits, topk_idx, part_p, part_cnt, status);
  router_stats_final_kernel<<<1, kFinalWarps * 32, 0, stream>>>(
      T, E, k, blocks, alpha, part_p, part_cnt, f, P, counts_routed, aux_loss);
  return launch_status();
}

// b_e += gamma if expert e's routed load is below the mean T*k/E, -= gamma
// if above, unchanged if equal (exact integer comparison).
__global__ void router_bias_update_kernel(int T, int E, int k, float gamma,
                                          const int32_t* __restrict__ counts,
                                          float* __restrict__ bias) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t d = static_cast<int64_t>(T) * k -
                    static_cast<int64_t>(E) * counts[e];
  if (d > 0)
    bias[e] = __fadd_rn(bias[e], gamma);
  else if (d < 0)
    bias[e] = __fsub_rn(bias[e], gamma);
}

moe_status launch_router_bias_update(int T, int E, int k, float gamma,
                                     const int32_t* counts, float* bias,
                                     cudaStream_t stream) {
  router_bias_update_kernel<<<static_cast<unsigned>(ceil_div(E, 256)), 256, 0,
                              stream>>>(T, E, k, gamma, counts, bias);
  return launch_status();
}

}  // namespace moe
