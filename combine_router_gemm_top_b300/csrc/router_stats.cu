// Router statistics of one routing decision ("Expert Parallelism in LLMs",
// Static Capacity Factors and Token Dropping: the auxiliary load-balancing
// loss L_aux = alpha * E * sum_i f_i * P_i, f_i the fraction of routed
// pairs on expert i, P_i the mean router probability of expert i) and the
// auxiliary-loss-free bias step (same page, Modern Dropless Dynamic
// Dispatch: bias terms on the routing scores adjusted to keep the load
// balanced).
//
// One memset and one kernel.  Each warp takes tokens, evaluates the router
// probabilities in fp32 and rounds each to a multiple of 2^-32; warps add
// their sums into the block's shared uint64 accumulators, and blocks add
// theirs into global ones.  The sums are exact 64-bit integers (below 2^63
// for T < 2^31; the error on P_e is below 2^-33), so they do not depend on
// the order of the additions and the results are deterministic.  Routed
// counts are added the same way.  The last block to finish forms f, P and
// L_aux, adding f_i * P_i through a fixed tree.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kStatsWarps = 8;
constexpr float kFix = 4294967296.0f;          // 2^32
constexpr double kInvFix = 1.0 / 4294967296.0;

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

struct StatsAcc {
  unsigned long long p[256];   // sum of p_e in units of 2^-32
  unsigned int cnt[256];       // routed pairs of expert e
  unsigned int done;           // blocks finished
};

// One warp per token (grid-stride); lane l holds experts l + 32 i.
template <int NI>
__global__ void __launch_bounds__(kStatsWarps * 32)
    router_stats_kernel(int T, int E, int k, int score, float alpha,
                        const float* __restrict__ logits,
                        const int32_t* __restrict__ topk_idx,
                        StatsAcc* __restrict__ acc_g, float* __restrict__ f,
                        float* __restrict__ P,
                        int32_t* __restrict__ counts_routed,
                        float* __restrict__ aux_loss, int32_t* status) {
  __shared__ unsigned long long s_p[NI * 32];
  __shared__ unsigned int s_cnt[NI * 32];
  __shared__ unsigned int s_ticket;
  __shared__ double s_fp[kStatsWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < NI * 32; i += blockDim.x) {
    s_p[i] = 0ull;
    s_cnt[i] = 0u;
  }
  __syncthreads();

  unsigned long long acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0ull;
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
    for (int i = 0; i < NI; ++i) acc[i] += __float2ull_rn(p[i] * kFix);
    if (lane < k) {
      const int e = topk_idx[t * k + lane];
      if (e >= 0 && e < E)
        atomicAdd(&s_cnt[e], 1u);
      else
        set_status(status, MOE_ERR_INDEX);
    }
  }
#pragma unroll
  for (int i = 0; i < NI; ++i)
    if (lane + 32 * i < E && acc[i] != 0ull) atomicAdd(&s_p[lane + 32 * i], acc[i]);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (s_p[e] != 0ull) atomicAdd(&acc_g->p[e], s_p[e]);
    if (s_cnt[e] != 0u) atomicAdd(&acc_g->cnt[e], s_cnt[e]);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(&acc_g->done, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;

  // the last block: every block's additions are visible
  __threadfence();
  const double pairs = static_cast<double>(T) * k;
  double fp = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const unsigned long long sum = atomicAdd(&acc_g->p[e], 0ull);
    const unsigned int cnt = atomicAdd(&acc_g->cnt[e], 0u);
    const double fe = pairs > 0 ? static_cast<double>(cnt) / pairs : 0.0;
    const double pe =
        T > 0 ? static_cast<double>(sum) * kInvFix / static_cast<double>(T)
              : 0.0;
    f[e] = static_cast<float>(fe);
    P[e] = static_cast<float>(pe);
    if (counts_routed != nullptr) counts_routed[e] = static_cast<int32_t>(cnt);
    fp += fe * pe;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) fp += __shfl_xor_sync(0xffffffffu, fp, d);
  if (lane == 0) s_fp[warp] = fp;
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int w = 0; w < kStatsWarps; ++w) sum += s_fp[w];
    aux_loss[0] = static_cast<float>(static_cast<double>(alpha) * E * sum);
  }
}

size_t router_stats_ws_bytes(int T, int E) {
  (void)T;
  (void)E;
  return sizeof(StatsAcc);
}

moe_status launch_router_stats(int T, int E, int k, int score,
                               const float* logits, const int32_t* topk_idx,
                               float alpha, float* f, float* P,
                               int32_t* counts_routed, float* aux_loss,
                               void* ws, int32_t* status,
                               cudaStream_t stream) {
  StatsAcc* acc = static_cast<StatsAcc*>(ws);
  if (cudaMemsetAsync(acc, 0, sizeof(StatsAcc), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  // one token per warp up to 4 blocks per SM, then a grid-stride loop
  const int64_t want = ceil_div(T, kStatsWarps);
  const int64_t cap = 4 * kNumSMs;
  const unsigned blocks =
      static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
  const int ni = static_cast<int>(ceil_div(E, 32));
  const dim3 block(kStatsWarps * 32);
  if (ni <= 1)
    router_stats_kernel<1><<<blocks, block, 0, stream>>>(
        T, E, k, score, alpha, logits, topk_idx, acc, f, P, counts_routed,
        aux_loss, status);
  else if (ni <= 2)
    router_stats_kernel<2><<<blocks, block, 0, stream>>>(
        T, E, k, score, alpha, logits, topk_idx, acc, f, P, counts_routed,
        aux_loss, status);
  else if (ni <= 4)
    router_stats_kernel<4><<<blocks, block, 0, stream>>>(
        T, E, k, score, alpha, logits, topk_idx, acc, f, P, counts_routed,
        aux_loss, status);
  else
    router_stats_kernel<8><<<blocks, block, 0, stream>>>(
        T, E, k, score, alpha, logits, topk_idx, acc, f, P, counts_routed,
        aux_loss, status);
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
