// Backward pass of the MoE layer, the row movers and the router
// ("Expert Parallelism in LLMs", Backward Pass Symmetry: the upstream
// gradient dL/dy goes to the experts along the dispatch pattern, the input
// gradients return along the combine pattern).  The routing decision is
// held fixed; gradients flow through the gates and the experts.
//
//   combine backward  dYp[row(t,j)] = g[t,j] * dy[t] and
//                     dgate[t,j] = dy[t] . Yp[row(t,j)] (fp32, 0 if dropped)
//   permute backward  dx[t] = sum over kept j of dXp[row(t,j)] (the combine
//                     kernel with unit gates)
//   aligned layout    expert segments moved to 64-row boundaries so that the
//                     weight-gradient GEMMs, which contract over an expert's
//                     token rows, never reach into the next expert; padding
//                     rows are zero
//   router backward   dlogits from dgate per score mode, dW_r = dlogits^T x,
//                     dx += dlogits W_r (fp32 accumulation, fixed order)
#include <float.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "umma_gemm.cuh"

namespace moe {

constexpr int kBwdWarps = 8;

__device__ __forceinline__ float bwd_warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// ------------------------------------------------------ combine backward
// One warp per token.  For each kept slot: the gate-scaled copy of dy[t]
// into the slot's expert row and the dot product of dy[t] with the expert
// output row.  dy[t] is re-read per slot from L1/L2.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32)
    combine_backward_kernel(int64_t n_tok, int k, int nvec,
                            const uint4* __restrict__ dy,
                            const uint4* __restrict__ yp,
                            const int32_t* __restrict__ dst_row,
                            const float* __restrict__ gate,
                            uint4* __restrict__ dyp,
                            float* __restrict__ dgate, int max_rows,
                            int32_t* status) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kBwdWarps;
  for (int64_t t = w0; t < n_tok; t += nw) {
    const int32_t my_dst = checked_row(
        lane < k ? __ldg(dst_row + t * k + lane) : -1, max_rows, status);
    const float my_g = lane < k ? __ldg(gate + t * k + lane) : 0.0f;
    const uint4* src = dy + t * nvec;
    float my_dot = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int32_t r = __shfl_sync(0xffffffffu, my_dst, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      if (r < 0) continue;
      const uint4* yrow = yp + static_cast<int64_t>(r) * nvec;
      uint4* drow = dyp + static_cast<int64_t>(r) * nvec;
      float dot = 0.0f;
      for (int v = lane; v < nvec; v += 32) {
        float a[N], b[N], o[N];
        Vec16<T>::to_f32(ld_nc_v4(src + v), a);
        Vec16<T>::to_f32(ld_nc_v4(yrow + v), b);
#pragma unroll
        for (int i = 0; i < N; ++i) {
          dot = fmaf(a[i], b[i], dot);
          o[i] = g * a[i];
        }
        st_v4(drow + v, Vec16<T>::from_f32(o));
      }
      dot = bwd_warp_sum(dot);
      if (lane == j) my_dot = dot;
    }
    if (lane < k) dgate[t * k + lane] = my_dst >= 0 ? my_dot : 0.0f;
  }
}

moe_status launch_combine_backward(int T, int k, int D, int dtype,
                                   const void* dy, const void* yp,
                                   const int32_t* dst_row, const float* gate,
                                   void* dyp, float* dgate, int max_rows,
                                   int32_t* status, cudaStream_t stream,
                                   int num_sms) {
  if (T == 0) return MOE_OK;
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  const int64_t want = ceil_div(T, kBwdWarps);
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (dtype == MOE_BF16)
    combine_backward_kernel<__nv_bfloat16><<<grid, kBwdWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(dy),
        static_cast<const uint4*>(yp), dst_row, gate,
        static_cast<uint4*>(dyp), dgate, max_rows, status);
  else
    combine_backward_kernel<float><<<grid, kBwdWarps * 32, 0, stream>>>(
        T, k, nvec, static_cast<const uint4*>(dy),
        static_cast<const uint4*>(yp), dst_row, gate,
        static_cast<uint4*>(dyp), dgate, max_rows, status);
  return launch_status();
}

// ------------------------------------------------------ aligned layout
// One block: offsets_aligned = exclusive scan of round_up(count_e, align).
__global__ void __launch_bounds__(1024)
    aligned_offsets_kernel(int E, int align, const int32_t* __restrict__ off,
                           int32_t* __restrict__ off_a) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < E; base += 1024) {
    const int e = base + threadIdx.x;
    int v = 0;
    if (e < E) {
      const int c = __ldg(off + e + 1) - __ldg(off + e);
      v = (c + align - 1) / align * align;
    }
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
      int wi = w;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, wi, d);
        if (lane >= d) wi += u;
      }
      warp_tot[lane] = wi - w;   // exclusive prefix of warp totals
    }
    __syncthreads();
    const int c0 = carry;
    if (e < E) off_a[e] = c0 + warp_tot[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == 1023) carry = c0 + warp_tot[31] + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) off_a[E] = carry;
}

__global__ void aligned_rows_kernel(int64_t P, int E,
                                    const int32_t* __restrict__ topk_idx,
                                    const int32_t* __restrict__ dst_row,
                                    const int32_t* __restrict__ off,
                                    const int32_t* __restrict__ off_a,
                                    int32_t* __restrict__ dst_a,
                                    int32_t* status) {
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= P) return;
  const int r = __ldg(dst_row + p);
  int out = -1;
  if (r >= 0) {
    const int e = __ldg(topk_idx + p);
    if (e >= 0 && e < E)
      out = __ldg(off_a + e) + (r - __ldg(off + e));
    else
      set_status(status, MOE_ERR_INDEX);
  }
  dst_a[p] = out;
}

moe_status launch_aligned_layout(int T, int k, int E, int align,
                                 const int32_t* topk_idx,
                                 const int32_t* dst_row,
                                 const int32_t* offsets,
                                 int32_t* dst_row_aligned,
                                 int32_t* offsets_aligned, int32_t* status,
                                 cudaStream_t stream) {
  aligned_offsets_kernel<<<1, 1024, 0, stream>>>(E, align, offsets,
                                                 offsets_aligned);
  const int64_t P = static_cast<int64_t>(T) * k;
  if (P > 0)
    aligned_rows_kernel<<<static_cast<unsigned>(ceil_div(P, 256)), 256, 0,
                          stream>>>(P, E, topk_idx, dst_row, offsets,
                                    offsets_aligned, dst_row_aligned, status);
  return launch_status();
}

// Zero rows [off_a[e] + count_e, off_a[e+1]) of every expert: one block per
// expert, one warp per padding row.
__global__ void __launch_bounds__(256)
    aligned_fill_kernel(int nvec, const int32_t* __restrict__ off,
                        const int32_t* __restrict__ off_a,
                        uint4* __restrict__ buf) {
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int r0 = __ldg(off_a + e) + (__ldg(off + e + 1) - __ldg(off + e));
  const int r1 = __ldg(off_a + e + 1);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int r = r0 + (threadIdx.x >> 5); r < r1; r += 8) {
    uint4* row = buf + static_cast<int64_t>(r) * nvec;
    for (int v = lane; v < nvec; v += 32) st_v4(row + v, z);
  }
}

moe_status launch_aligned_fill(int E, int D, int dtype, const int32_t* offsets,
                               const int32_t* offsets_aligned, void* buf,
                               cudaStream_t stream) {
  const int nvec = static_cast<int>(D * dtype_bytes(dtype) / 16);
  aligned_fill_kernel<<<static_cast<unsigned>(E), 256, 0, stream>>>(
      nvec, offsets, offsets_aligned, static_cast<uint4*>(buf));
  return launch_status();
}

// ------------------------------------------------------ router backward
// One warp per token; lane l holds experts l + 32 i.  Slot j's id, gate
// gradient and logit live in lane j (k <= 32).
template <int NI>
__global__ void __launch_bounds__(kBwdWarps * 32)
    dlogits_kernel(int T, int E, int k, int score,
                   const float* __restrict__ logits,
                   const int32_t* __restrict__ topk_idx,
                   const float* __restrict__ dgate,
                   float* __restrict__ dlogits,
                   __nv_bfloat16* __restrict__ dl2) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const bool slot = lane < k;
  const int my_e = slot ? topk_idx[t * k + lane] : -1;
  const float my_dg = slot ? dgate[t * k + lane] : 0.0f;
  const bool my_ok = slot && my_e >= 0 && my_e < E;
  const float my_l = my_ok ? logits[t * E + my_e] : 0.0f;
  float out[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) out[i] = 0.0f;

  if (score == MOE_SCORE_SOFTMAX_FULL) {
    // g_j = p_{e_j}, p = softmax over all E: dl = p (dp - p . dp)
    float l[NI], p[NI], dp[NI];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      l[i] = e < E ? logits[t * E + e] : -FLT_MAX;
      m = fmaxf(m, l[i]);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      p[i] = lane + 32 * i < E ? expf(l[i] - m) : 0.0f;
      z += p[i];
      dp[i] = 0.0f;
    }
    z = bwd_warp_sum(z);
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_ok ? my_e : -1, j);
      const float gj = __shfl_sync(0xffffffffu, my_dg, j);
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (lane + 32 * i == ej) dp[i] += gj;
    }
    float pdp = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      p[i] = p[i] / z;
      pdp += p[i] * dp[i];
    }
    pdp = bwd_warp_sum(pdp);
#pragma unroll
    for (int i = 0; i < NI; ++i) out[i] = p[i] * (dp[i] - pdp);
  } else {
    float dl_slot = 0.0f;
    if (score == MOE_SCORE_SOFTMAX_TOPK) {
      // g = softmax over the selected logits: dl_j = g_j (dg_j - g . dg)
      float m = my_ok ? my_l : -FLT_MAX;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
      const float ex = my_ok ? expf(my_l - m) : 0.0f;
      const float g = ex / bwd_warp_sum(ex);
      const float gdg = bwd_warp_sum(g * my_dg);
      dl_slot = g * (my_dg - gdg);
    } else {
      // g_j = s_j / S over the selected sigmoid scores:
      // dl_j = (dg_j - g . dg) / S * s_j (1 - s_j)
      const float s = my_ok ? 1.0f / (1.0f + expf(-my_l)) : 0.0f;
      const float S = bwd_warp_sum(s);
      const float g = s / S;
      const float gdg = bwd_warp_sum(g * my_dg);
      dl_slot = (my_dg - gdg) / S * s * (1.0f - s);
    }
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_ok ? my_e : -1, j);
      const float dj = __shfl_sync(0xffffffffu, dl_slot, j);
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (lane + 32 * i == ej) out[i] += dj;
    }
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      dlogits[t * E + e] = out[i];
      if (dl2 != nullptr) {
        // two bf16 terms: hi = bf16(dl), lo = bf16(dl - hi) (the difference
        // is exact in fp32)
        const __nv_bfloat16 hi = __float2bfloat16_rn(out[i]);
        const __nv_bfloat16 lo =
            __float2bfloat16_rn(out[i] - __bfloat162float(hi));
        dl2[t * 2 * E + e] = hi;
        dl2[t * 2 * E + E + e] = lo;
      }
    }
  }
}

// dW_r[e, d] = sum_t dl[t, e] x[t, d].  Block = 256 columns d x EB experts
// over one slice of the tokens; slices are summed in a fixed order by
// dwr_reduce_kernel (or written directly when there is one slice).
template <typename T, int EB>
__global__ void __launch_bounds__(256)
    dwr_kernel(int Tn, int E, int D, int t_per_slice,
               const float* __restrict__ dl, const T* __restrict__ x,
               float* __restrict__ out) {
  __shared__ float s_dl[32][EB];
  const int d = blockIdx.x * 256 + threadIdx.x;
  const int e0 = blockIdx.y * EB;
  const int ts = blockIdx.z * t_per_slice;
  const int te = min(Tn, ts + t_per_slice);
  float acc[EB];
#pragma unroll
  for (int i = 0; i < EB; ++i) acc[i] = 0.0f;
  for (int t0 = ts; t0 < te; t0 += 32) {
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * EB; i += 256) {
      const int tt = t0 + i / EB, ee = e0 + i % EB;
      s_dl[i / EB][i % EB] =
          tt < te && ee < E ? dl[static_cast<int64_t>(tt) * E + ee] : 0.0f;
    }
    __syncthreads();
    if (d < D) {
      const int tn = min(32, te - t0);
      for (int i = 0; i < tn; ++i) {
        const float xv =
            static_cast<float>(x[static_cast<int64_t>(t0 + i) * D + d]);
#pragma unroll
        for (int j = 0; j < EB; ++j) acc[j] = fmaf(s_dl[i][j], xv, acc[j]);
      }
    }
  }
  if (d < D) {
    float* o = out + static_cast<int64_t>(blockIdx.z) * E * D;
#pragma unroll
    for (int j = 0; j < EB; ++j)
      if (e0 + j < E) o[static_cast<int64_t>(e0 + j) * D + d] = acc[j];
  }
}

// dW_r for E >= 64 (bf16 x): block = 64 experts x 256 columns over one
// token slice; thread = 8 experts x 8 columns, 64 accumulators.  16 tokens
// of x (fp32) and dl sit in shared memory per step; each token costs a
// thread 4 shared float4 loads for 64 FMAs.
__global__ void __launch_bounds__(256)
    dwr_tiled_kernel(int Tn, int E, int D, int t_per_slice,
                     const float* __restrict__ dl,
                     const __nv_bfloat16* __restrict__ x,
                     float* __restrict__ out) {
  __shared__ __align__(16) float s_x[16][256];
  __shared__ __align__(16) float s_l[16][64];
  const int tid = threadIdx.x;
  const int te = tid >> 5;          // experts e0 + 8*te .. +7
  const int td = tid & 31;          // columns d0 + 8*td .. +7
  const int e0 = blockIdx.y * 64;
  const int d0 = blockIdx.x * 256;
  const int ts = blockIdx.z * t_per_slice;
  const int tend = min(Tn, ts + t_per_slice);
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  for (int t0 = ts; t0 < tend; t0 += 16) {
    __syncthreads();
    // 16 tokens x 256 columns: 512 vectors of 8 bf16, two per thread
    for (int v = tid; v < 512; v += 256) {
      const int tt = v >> 5, dd = (v & 31) * 8;
      const int t = t0 + tt, d = d0 + dd;
      float f[8];
      if (t < tend && d < D) {
        Vec16<__nv_bfloat16>::to_f32(
            ld_nc_v4(x + static_cast<int64_t>(t) * D + d), f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.0f;
      }
      *reinterpret_cast<float4*>(&s_x[tt][dd]) =
          make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&s_x[tt][dd + 4]) =
          make_float4(f[4], f[5], f[6], f[7]);
    }
    for (int i = tid; i < 16 * 64; i += 256) {
      const int tt = i >> 6, ee = i & 63;
      const int t = t0 + tt, e = e0 + ee;
      s_l[tt][ee] =
          t < tend && e < E ? dl[static_cast<int64_t>(t) * E + e] : 0.0f;
    }
    __syncthreads();
#pragma unroll 4
    for (int tt = 0; tt < 16; ++tt) {
      const float4 l0 = *reinterpret_cast<const float4*>(&s_l[tt][8 * te]);
      const float4 l1 = *reinterpret_cast<const float4*>(&s_l[tt][8 * te + 4]);
      const float4 x0 = *reinterpret_cast<const float4*>(&s_x[tt][8 * td]);
      const float4 x1 = *reinterpret_cast<const float4*>(&s_x[tt][8 * td + 4]);
      const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
      const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(lv[i], xv[j], acc[i][j]);
    }
  }
  float* o = out + static_cast<int64_t>(blockIdx.z) * E * D;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e0 + 8 * te + i;
    const int d = d0 + 8 * td;
    if (e < E && d < D) {
      float* p = o + static_cast<int64_t>(e) * D + d;
      *reinterpret_cast<float4*>(p) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(p + 4) =
          make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
  }
}

__global__ void dwr_reduce_kernel(int64_t n, int slices,
                                  const float* __restrict__ part,
                                  float* __restrict__ dwr) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.0f;
  for (int k = 0; k < slices; ++k) s += part[k * n + i];
  dwr[i] = s;
}

// dx[t, d] += sum_e dl[t, e] W_r[e, d]: block = 256 columns d x 32 tokens.
// The block's dl values sit in shared memory expert-major, 32 tokens (plus
// 4 floats of padding) per expert, so each thread reads them as float4.
constexpr int kDxLd = 36;

template <typename T>
__global__ void __launch_bounds__(256)
    dx_router_kernel(int Tn, int E, int D, const float* __restrict__ dl,
                     const T* __restrict__ wr, T* __restrict__ dx) {
  extern __shared__ float s_dlt[];   // [E][kDxLd]
  const int d = blockIdx.x * 256 + threadIdx.x;
  const int t0 = blockIdx.y * 32;
  for (int i = threadIdx.x; i < 32 * E; i += 256) {
    const int tt = i / E, ee = i - tt * E;
    s_dlt[ee * kDxLd + tt] =
        t0 + tt < Tn ? dl[static_cast<int64_t>(t0 + tt) * E + ee] : 0.0f;
  }
  __syncthreads();
  if (d >= D) return;
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
#pragma unroll 4
  for (int e = 0; e < E; ++e) {
    const float w = static_cast<float>(wr[static_cast<int64_t>(e) * D + d]);
    const float4* q = reinterpret_cast<const float4*>(s_dlt + e * kDxLd);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = q[j];
      acc[4 * j] = fmaf(v.x, w, acc[4 * j]);
      acc[4 * j + 1] = fmaf(v.y, w, acc[4 * j + 1]);
      acc[4 * j + 2] = fmaf(v.z, w, acc[4 * j + 2]);
      acc[4 * j + 3] = fmaf(v.w, w, acc[4 * j + 3]);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int tt = t0 + j;
    if (tt < Tn) {
      T* p = dx + static_cast<int64_t>(tt) * D + d;
      *p = static_cast<T>(static_cast<float>(*p) + acc[j]);
    }
  }
}

// Token slices for dW_r: enough blocks to cover the SMs twice.
struct DwrPlan {
  int eb, slices, t_per_slice;
};
static DwrPlan dwr_plan(int T, int E, int D, int num_sms) {
  DwrPlan p;
  p.eb = E >= 64 ? 64 : (E >= 32 ? 32 : 8);
  const int64_t base = ceil_div(D, 256) * ceil_div(E, p.eb);
  // the tiled kernel keeps two blocks per SM resident: take as many slices
  // as fit in one round of them, not one more
  int64_t s = p.eb == 64 ? (2 * num_sms) / base : ceil_div(2 * num_sms, base);
  const int64_t max_s = ceil_div(T, 32);
  s = s < 1 ? 1 : (s > 64 ? 64 : s);
  s = s > max_s ? max_s : s;
  p.t_per_slice = static_cast<int>(ceil_div(ceil_div(T, s), 32) * 32);
  p.slices = static_cast<int>(ceil_div(T, p.t_per_slice));
  if (p.slices < 1) p.slices = 1;
  return p;
}

// Tensor-core router backward: bf16, E and D multiples of 64 (whole
// 64-wide boxes of dL2 and W_r, whole 32-column epilogue chunks).
bool route_bwd_tensor(int dtype, int E, int D) {
  return dtype == MOE_BF16 && E % 64 == 0 && D % 64 == 0;
}

struct RbwdPlan {
  int k_blocks;      // dW_r contraction blocks: hi and lo of each 64 tokens
  int splits, kb_per_split;
  size_t dl2_bytes;  // dL2 [T, 2E] bf16, rounded up to 256 bytes
};
static RbwdPlan rbwd_plan(int T, int E, int D, int num_sms) {
  RbwdPlan p;
  p.k_blocks = static_cast<int>(2 * ceil_div(T, kBK));
  const int64_t base = ceil_div(E, kBM) * ceil_div(D, 256);
  // fewest rounds of K blocks on the busiest SM; at most 8 splits so the
  // fp32 partials stay small
  int64_t best = INT64_MAX;
  p.kb_per_split = p.k_blocks;
  for (int s = 1; s <= 8; ++s) {
    const int kbps = static_cast<int>(ceil_div(p.k_blocks, s));
    const int64_t real_s = ceil_div(p.k_blocks, kbps);
    const int64_t cost = ceil_div(base * real_s, num_sms) * kbps;
    if (cost < best) {
      best = cost;
      p.kb_per_split = kbps;
    }
  }
  p.splits = static_cast<int>(ceil_div(p.k_blocks, p.kb_per_split));
  p.dl2_bytes = (static_cast<size_t>(T) * 2 * E * 2 + 255) & ~size_t(255);
  return p;
}

size_t route_bwd_ws_bytes(int T, int D, int E, int dtype, int num_sms) {
  if (route_bwd_tensor(dtype, E, D)) {
    const RbwdPlan p = rbwd_plan(T, E, D, num_sms);
    return p.dl2_bytes + (p.splits > 1 ? static_cast<size_t>(p.splits) * E *
                                             D * sizeof(float)
                                       : 0);
  }
  const DwrPlan p = dwr_plan(T, E, D, num_sms);
  return p.slices > 1 ? static_cast<size_t>(p.slices) * E * D * sizeof(float)
                      : 0;
}

bool route_bwd_uses_ws(int dtype, int E, int D, bool dw_r, bool dx) {
  return route_bwd_tensor(dtype, E, D) ? (dw_r || dx) : dw_r;
}

// dx += dL2 . [W_r; W_r] and dW_r = [hi; lo]^T . [x; x] on the tensor cores.
static moe_status launch_route_backward_tc(int T, int D, int E,
                                           const __nv_bfloat16* x,
                                           const __nv_bfloat16* w_r,
                                           const __nv_bfloat16* dl2,
                                           float* dw_r, __nv_bfloat16* dx,
                                           float* part, int32_t* status,
                                           cudaStream_t stream, int num_sms) {
  if (dx != nullptr) {
    CUtensorMap tm_dl, tm_w;
    if (!make_tmap_bf16_2d(&tm_dl, dl2, 2 * E, T, kBM) ||
        !make_tmap_bf16_2d(&tm_w, w_r, D, E, 64))
      return MOE_ERR_CUDA;
    GemmArgs g{};
    g.M = T;
    g.k_blocks = 2 * E / kBK;
    g.kb_per_split = g.k_blocks;
    g.splits = 1;
    g.BN = 256;
    g.stages = 4;
    g.tmem_cols = 512;
    g.E = E;
    g.n_tiles = static_cast<int>(ceil_div(D, 256));
    g.out = dx;
    g.out_ld = D;
    g.out_cols = D;
    g.status = status;
    g.wait_limit_ns = kWaitLimitNs;
    const moe_status st = launch_umma<kRDX>(tm_dl, tm_w, g, stream, num_sms);
    if (st != MOE_OK) return st;
  }
  if (dw_r != nullptr) {
    const RbwdPlan p = rbwd_plan(T, E, D, num_sms);
    CUtensorMap tm_dl, tm_x;
    if (!make_tmap_bf16_2d(&tm_dl, dl2, 2 * E, T, 64) ||
        !make_tmap_bf16_2d(&tm_x, x, D, T, 64))
      return MOE_ERR_CUDA;
    GemmArgs g{};
    g.M = E;
    g.k_blocks = p.k_blocks;
    g.kb_per_split = p.kb_per_split;
    g.splits = p.splits;
    g.BN = 256;
    g.stages = 3;
    g.tmem_cols = 512;
    g.E = E;
    g.n_tiles = static_cast<int>(ceil_div(D, 256));
    g.out = p.splits > 1 ? part : dw_r;
    g.out_ld = D;
    g.out_cols = D;
    g.row_limit = E;
    g.split_stride = static_cast<int64_t>(E) * D;
    g.status = status;
    g.wait_limit_ns = kWaitLimitNs;
    const moe_status st = launch_umma<kRDW>(tm_dl, tm_x, g, stream, num_sms);
    if (st != MOE_OK) return st;
    if (p.splits > 1) {
      const int64_t n = static_cast<int64_t>(E) * D;
      dwr_reduce_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                          stream>>>(n, p.splits, part, dw_r);
    }
  }
  return launch_status();
}

template <typename T>
static void launch_dwr(const DwrPlan& p, int Tn, int E, int D,
                       const float* dl, const T* x, float* dwr, float* ws,
                       cudaStream_t stream) {
  float* out = p.slices > 1 ? ws : dwr;
  const dim3 g(static_cast<unsigned>(ceil_div(D, 256)),
               static_cast<unsigned>(ceil_div(E, p.eb)),
               static_cast<unsigned>(p.slices));
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    if (p.eb == 64) {
      dwr_tiled_kernel<<<g, 256, 0, stream>>>(Tn, E, D, p.t_per_slice, dl, x,
                                              out);
    } else if (p.eb == 32) {
      dwr_kernel<T, 32><<<g, 256, 0, stream>>>(Tn, E, D, p.t_per_slice, dl, x, out);
    } else {
      dwr_kernel<T, 8><<<g, 256, 0, stream>>>(Tn, E, D, p.t_per_slice, dl, x, out);
    }
  } else {
    if (p.eb >= 32)
      dwr_kernel<T, 32><<<g, 256, 0, stream>>>(Tn, E, D, p.t_per_slice, dl, x, out);
    else
      dwr_kernel<T, 8><<<g, 256, 0, stream>>>(Tn, E, D, p.t_per_slice, dl, x, out);
  }
  if (p.slices > 1) {
    const int64_t n = static_cast<int64_t>(E) * D;
    dwr_reduce_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                        stream>>>(n, p.slices, ws, dwr);
  }
}

moe_status launch_route_backward(int T, int D, int E, int k, int score,
                                 int dtype, const void* x, const void* w_r,
                                 const float* logits, const int32_t* topk_idx,
                                 const float* dgate, float* dlogits,
                                 float* dw_r, void* dx, void* ws,
                                 int32_t* status, cudaStream_t stream,
                                 int num_sms) {
  if (T == 0) return MOE_OK;
  const bool tc = route_bwd_tensor(dtype, E, D) &&
                  (dw_r != nullptr || dx != nullptr);
  __nv_bfloat16* dl2 = tc ? static_cast<__nv_bfloat16*>(ws) : nullptr;
  const unsigned g1 = static_cast<unsigned>(ceil_div(T, kBwdWarps));
  const int ni = static_cast<int>(ceil_div(E, 32));
  if (ni <= 1)
    dlogits_kernel<1><<<g1, kBwdWarps * 32, 0, stream>>>(T, E, k, score, logits, topk_idx, dgate, dlogits, dl2);
  else if (ni <= 2)
    dlogits_kernel<2><<<g1, kBwdWarps * 32, 0, stream>>>(T, E, k, score, logits, topk_idx, dgate, dlogits, dl2);
  else if (ni <= 4)
    dlogits_kernel<4><<<g1, kBwdWarps * 32, 0, stream>>>(T, E, k, score, logits, topk_idx, dgate, dlogits, dl2);
  else
    dlogits_kernel<8><<<g1, kBwdWarps * 32, 0, stream>>>(T, E, k, score, logits, topk_idx, dgate, dlogits, dl2);
  if (tc) {
    const RbwdPlan p = rbwd_plan(T, E, D, num_sms);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                           p.dl2_bytes);
    return launch_route_backward_tc(
        T, D, E, static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(w_r), dl2, dw_r,
        static_cast<__nv_bfloat16*>(dx), part, status, stream, num_sms);
  }
  const DwrPlan p = dwr_plan(T, E, D, num_sms);
  const dim3 gx(static_cast<unsigned>(ceil_div(D, 256)),
                static_cast<unsigned>(ceil_div(T, 32)));
  const size_t smem = static_cast<size_t>(kDxLd) * E * sizeof(float);
  if (dtype == MOE_BF16) {
    if (dw_r != nullptr)
      launch_dwr(p, T, E, D, dlogits, static_cast<const __nv_bfloat16*>(x),
                 dw_r, static_cast<float*>(ws), stream);
    if (dx != nullptr)
      dx_router_kernel<__nv_bfloat16><<<gx, 256, smem, stream>>>(
          T, E, D, dlogits, static_cast<const __nv_bfloat16*>(w_r),
          static_cast<__nv_bfloat16*>(dx));
  } else {
    if (dw_r != nullptr)
      launch_dwr(p, T, E, D, dlogits, static_cast<const float*>(x), dw_r,
                 static_cast<float*>(ws), stream);
    if (dx != nullptr)
      dx_router_kernel<float><<<gx, 256, smem, stream>>>(
          T, E, D, dlogits, static_cast<const float*>(w_r),
          static_cast<float*>(dx));
  }
  return launch_status();
}

}  // namespace moe
