// moe_route kernels: router GEMM (tcgen05 split-K for bf16, fp32 FMA for
// fp32), then per-token scoring, group-limited top-k and gates
// ("Expert Parallelism in LLMs", The Execution Pipeline, step 1 "Router
// Gating and Softmax Selection": g_t = Softmax(TopK(W_g x_t, k))).
#include <cuda.h>
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "umma_gemm.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// fp32 sigmoid used for selection keys.  Selection is an integer decision
// taken on fp32 values, so both this library and any checker must evaluate
// the key with the same fp32 operations.  The recipe (Cody-Waite range
// reduction, W. J. Cody and W. Waite, "Software Manual for the Elementary
// Functions", 1980, followed by the degree-7 Taylor polynomial of exp on
// |r| <= ln2/2 in Horner form), every step one IEEE round-to-nearest fp32
// operation with no fused multiply-add:
//   z  = clamp(-l, -87, 88)
//   n  = rint(z * LOG2E)
//   r  = (z - n*LN2_HI) - n*LN2_LO          (n*LN2_HI is exact)
//   p  = c7; p = p*r + c_i for i = 6..0      (c_i = fp32(1/i!))
//   e  = p * 2^n                             (exact: the result is normal)
//   s  = 1 / (1 + e)
// LN2_HI is ln 2 in fp32 with the low 12 mantissa bits cleared, LN2_LO the
// fp32 rounding of the remainder.  Maximum error against the exact sigmoid
// is a few fp32 ulp.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sigmoid_key_f32(float l) {
  const float kLog2e = 1.44269502162933349609375f;   // 0x3FB8AA3B
  const float kLn2Hi = 0.693115234375f;              // 0x3F317000
  const float kLn2Lo = 3.194618329871446e-05f;       // 0x3805FDF4
  const float c[8] = {1.0f, 1.0f, 0.5f, 0.1666666716337204f,
                      0.0416666679084301f, 0.008333333767950535f,
                      0.0013888889225199819f, 0.00019841270113829523f};
  float z = -l;
  z = fminf(fmaxf(z, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(z, kLog2e));
  const float r = __fsub_rn(__fsub_rn(z, __fmul_rn(n, kLn2Hi)),
                            __fmul_rn(n, kLn2Lo));
  float p = c[7];
#pragma unroll
  for (int i = 6; i >= 0; --i) p = __fadd_rn(__fmul_rn(p, r), c[i]);
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

struct KeyIdx {
  float key;
  int idx;
};
// a beats b: larger key, or equal key and lower index
__device__ __forceinline__ bool beats(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}
__device__ __forceinline__ KeyIdx warp_best(KeyIdx v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, v.key, d);
    const int oi = __shfl_xor_sync(0xffffffffu, v.idx, d);
    if (beats(ok, oi, v.key, v.idx)) {
      v.key = ok;
      v.idx = oi;
    }
  }
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// One warp per token; lane l holds experts e = l + 32*i, i < NI.
template <int NI>
__global__ void __launch_bounds__(256)
    route_select_kernel(RouteSelectArgs a) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int E = a.E;

  float lg[NI], key[NI];
  bool elig[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    elig[i] = e < E;
    float l = 0.0f;
    if (elig[i]) {
      // split-K partial sums added in split order
      l = a.partial[t * E + e];
      for (int s = 1; s < a.splits; ++s)
        l = __fadd_rn(l, a.partial[(static_cast<int64_t>(s) * a.T + t) * E + e]);
      if (a.logit_offset != nullptr) l = __fadd_rn(l, a.logit_offset[e]);
      if (a.logits_out != nullptr) a.logits_out[t * E + e] = l;
    }
    lg[i] = l;
    float k = l;
    if (a.score == MOE_SCORE_SIGMOID_BIAS && elig[i]) {
      k = sigmoid_key_f32(l);
      if (a.sel_bias != nullptr) k = __fadd_rn(k, a.sel_bias[e]);
    }
    key[i] = k;
  }

  // group-limited selection: keep the topk_groups best groups
  if (a.n_groups > 1) {
    const int gs = E / a.n_groups;
    float my_gscore = -FLT_MAX;   // lane g holds group g's score
    for (int g = 0; g < a.n_groups; ++g) {
      uint32_t taken = 0;        // per-lane bitmask over its NI slots
      float acc = 0.0f;
      for (int j = 0; j < a.group_score_topk; ++j) {
        KeyIdx best{-INFINITY, 0x7fffffff};
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int e = lane + 32 * i;
          if (elig[i] && e / gs == g && !((taken >> i) & 1u) &&
              beats(key[i], e, best.key, best.idx)) {
            best.key = key[i];
            best.idx = e;
          }
        }
        best = warp_best(best);
        acc = __fadd_rn(acc, best.key);
#pragma unroll
        for (int i = 0; i < NI; ++i)
          if (lane + 32 * i == best.idx) taken |= 1u << i;
      }
      if (lane == g) my_gscore = acc;
    }
    uint32_t chosen = 0;
    bool gtaken = false;
    for (int j = 0; j < a.topk_groups; ++j) {
      KeyIdx c{(lane < a.n_groups && !gtaken) ? my_gscore : -INFINITY,
               (lane < a.n_groups && !gtaken) ? lane : 0x7fffffff};
      c = warp_best(c);
      chosen |= 1u << c.idx;
      if (lane == c.idx) gtaken = true;
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (elig[i] && !((chosen >> (e / gs)) & 1u)) elig[i] = false;
    }
  }

  // top-k by repeated warp arg-max; lane j keeps slot j
  int my_idx = -1;
  float my_logit = 0.0f;
  for (int j = 0; j < a.k; ++j) {
    KeyIdx best{-INFINITY, 0x7fffffff};
    float best_l = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (elig[i] && beats(key[i], e, best.key, best.idx)) {
        best.key = key[i];
        best.idx = e;
        best_l = lg[i];
      }
    }
    const KeyIdx w = warp_best(best);
    // the owner lane of the winner broadcasts its logit
    const int owner = w.idx & 31;
    const float wl = __shfl_sync(0xffffffffu, best_l, owner);
    if (lane == j) {
      my_idx = w.idx;
      my_logit = wl;
    }
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i == w.idx) elig[i] = false;
  }

  // gates
  const bool slot = lane < a.k;
  float g = 0.0f;
  if (a.score == MOE_SCORE_SOFTMAX_TOPK) {
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);   // slot 0 = max
    const float ex = slot ? expf(my_logit - m) : 0.0f;
    g = ex / warp_sum(ex);
  } else if (a.score == MOE_SCORE_SOFTMAX_FULL) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) m = fmaxf(m, lg[i]);
    m = warp_max(m);
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) z += expf(lg[i] - m);
    z = warp_sum(z);
    g = slot ? expf(my_logit - m) / z : 0.0f;
  } else {
    const float s = slot ? sigmoid_key_f32(my_logit) : 0.0f;
    g = s / warp_sum(s);
  }
  if (slot) {
    a.topk_idx[t * a.k + lane] = my_idx;
    a.topk_gate[t * a.k + lane] = g;
  }
}

// fp32 router GEMM on the FMA pipes: one thread per (token, expert).
__global__ void route_gemm_f32_kernel(int T, int D, int E, const float* x,
                                      const float* w, float* logits) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * E) return;
  const int64_t t = i / E;
  const int e = static_cast<int>(i - t * E);
  const float* xr = x + t * D;
  const float* wr = w + static_cast<int64_t>(e) * D;
  float acc = 0.0f;
  for (int d = 0; d < D; ++d) acc = fmaf(xr[d], wr[d], acc);
  logits[i] = acc;
}

__global__ void sigmoid_key_kernel(const float* l, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = sigmoid_key_f32(l[i]);
}

moe_status launch_sigmoid_key(const float* l, float* out, int n,
                              cudaStream_t stream) {
  if (n == 0) return MOE_OK;
  sigmoid_key_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                       stream>>>(l, out, n);
  return launch_status();
}

// ------------------------------------------------------------------ host
RoutePlan plan_route(const moe_route_cfg& c, int num_sms) {
  RoutePlan p{};
  p.Npad = ((c.E + 15) / 16) * 16;
  p.k_blocks = static_cast<int>(ceil_div(c.D, kBK));
  const int m_tiles = static_cast<int>(ceil_div(c.T, kBM));
  int splits = 1;
  if (c.dtype == MOE_BF16) {
    // enough (m block, K split) tiles to cover the SMs, >= 4 K blocks each
    splits = num_sms / (m_tiles > 0 ? m_tiles : 1);
    splits = splits < 1 ? 1 : splits;
    const int max_splits = p.k_blocks / 4 > 0 ? p.k_blocks / 4 : 1;
    splits = splits > max_splits ? max_splits : splits;
  }
  p.kb_per_split = static_cast<int>(ceil_div(p.k_blocks, splits));
  p.splits = static_cast<int>(ceil_div(p.k_blocks, p.kb_per_split));
  if (c.dtype != MOE_BF16) p.splits = 1;
  p.ws_bytes = static_cast<size_t>(p.splits) * c.T * c.E * sizeof(float);
  return p;
}

moe_status launch_route(const moe_route_cfg& c, const void* x, const void* w_r,
                        const float* logit_offset, const float* sel_bias,
                        int32_t* topk_idx, float* topk_gate, float* logits_out,
                        void* ws, int32_t* status, cudaStream_t stream,
                        int num_sms) {
  const RoutePlan p = plan_route(c, num_sms);
  float* partial = static_cast<float*>(ws);
  if (c.dtype == MOE_BF16) {
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16_2d(&tmA, x, c.D, c.T, kBM) ||
        !make_tmap_bf16_2d(&tmB, w_r, c.D, c.E, p.Npad))
      return MOE_ERR_CUDA;
    GemmArgs g{};
    g.M = c.T;
    g.k_blocks = p.k_blocks;
    g.BN = p.Npad;
    const size_t stage_bytes = kATileBytes + static_cast<size_t>(p.Npad) * kBK * 2;
    int stages = static_cast<int>((200 * 1024) / stage_bytes);
    g.stages = stages > kMaxStages ? kMaxStages : stages;
    int cols = 32;
    while (cols < 2 * p.Npad) cols <<= 1;
    g.tmem_cols = cols;
    g.splits = p.splits;
    g.kb_per_split = p.kb_per_split;
    g.E = c.E;
    g.out = partial;
    g.out_ld = c.E;
    g.out_cols = c.E;
    g.status = status;
    g.wait_limit_ns = kWaitLimitNs;
    const size_t smem = umma_gemm_smem_bytes(g.BN, g.stages);
    static bool attr_set = false;
    if (!attr_set) {
      if (cudaFuncSetAttribute(umma_gemm_kernel<kRoute>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024) != cudaSuccess)
        return MOE_ERR_CUDA;
      attr_set = true;
    }
    const int tiles = static_cast<int>(ceil_div(c.T, kBM)) * p.splits;
    const int grid = tiles < num_sms ? tiles : num_sms;
    umma_gemm_kernel<kRoute><<<grid, kGemmThreads, smem, stream>>>(tmA, tmB, g);
  } else {
    const int64_t n = static_cast<int64_t>(c.T) * c.E;
    route_gemm_f32_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                            stream>>>(c.T, c.D, c.E,
                                      static_cast<const float*>(x),
                                      static_cast<const float*>(w_r), partial);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  RouteSelectArgs s{};
  s.T = c.T;
  s.E = c.E;
  s.k = c.k;
  s.score = c.score;
  s.n_groups = c.n_groups;
  s.topk_groups = c.topk_groups;
  s.group_score_topk = c.group_score_topk;
  s.splits = p.splits;
  s.partial = partial;
  s.logit_offset = logit_offset;
  s.sel_bias = sel_bias;
  s.topk_idx = topk_idx;
  s.topk_gate = topk_gate;
  s.logits_out = logits_out;
  const int warps = 8;
  const unsigned grid = static_cast<unsigned>(ceil_div(c.T, warps));
  const int ni = static_cast<int>(ceil_div(c.E, 32));
  if (ni <= 1)
    route_select_kernel<1><<<grid, warps * 32, 0, stream>>>(s);
  else if (ni <= 2)
    route_select_kernel<2><<<grid, warps * 32, 0, stream>>>(s);
  else if (ni <= 4)
    route_select_kernel<4><<<grid, warps * 32, 0, stream>>>(s);
  else
    route_select_kernel<8><<<grid, warps * 32, 0, stream>>>(s);
  return launch_status();
}

}  // namespace moe
