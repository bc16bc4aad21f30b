// Internal host-side interfaces between the C-ABI layer (api.cu) and the
// kernel files.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Upper bound on any single wait inside a kernel (a stalled pipeline
// reports MOE_ERR_TIMEOUT instead of hanging the GPU).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box of 64
// columns (128 bytes, 128-byte swizzle) by box_rows rows; out-of-bounds
// elements read as zero.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t cols,
                       int64_t rows, int box_rows);

struct RoutePlan {
  int Npad;          // E rounded up to 16 (MMA N)
  int k_blocks;      // ceil(D / 64)
  int splits;        // split-K factor of the router GEMM
  int kb_per_split;
  size_t ws_bytes;   // partial logits [splits][T][E] fp32
};
RoutePlan plan_route(const moe_route_cfg& c, int num_sms);
bool route_single_kernel(const moe_route_cfg& c, int num_sms);
bool route_fused_gemm(const moe_route_cfg& c, int num_sms);

struct RouteSelectArgs {
  int T, E, k, score, n_groups, topk_groups, group_score_topk, splits;
  const float* partial;
  const float* logit_offset;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_gate;
  float* logits_out;
  int32_t* status;  // receives MOE_ERR_TIMEOUT if a bounded wait expires
};

moe_status launch_route(const moe_route_cfg& c, const void* x, const void* w_r,
                        const float* logit_offset, const float* sel_bias,
                        int32_t* topk_idx, float* topk_gate, float* logits_out,
                        void* ws, int32_t* status, cudaStream_t stream,
                        int num_sms);

constexpr int kLayoutChunk = 2048;   // pairs per layout block
constexpr int kLayoutMaxE = 1024;
constexpr int kMaxGroupsApi = 1024;   // experts the grouped tcgen05 scheduler handles
size_t layout_ws_bytes(int64_t P, int E);
int layout_launches(int64_t P, int E);
moe_status launch_layout(int T, int k, int E, int R, int capacity,
                         const int32_t* topk_idx, int32_t* expert_counts,
                         int32_t* expert_offsets, int32_t* dst_row,
                         int32_t* src_pair, int32_t* n_kept,
                         int32_t* n_dropped, int32_t* rank_send_counts,
                         int32_t* rank_send_displs, void* ws, int32_t* status,
                         cudaStream_t stream);

moe_status launch_permute(int T, int k, int D, int dtype, const void* x,
                          const int32_t* dst_row, void* xp, int max_rows,
                          int32_t* status, cudaStream_t stream, int num_sms);
moe_status launch_combine(int T, int k, int D, int dtype, const void* yp,
                          const int32_t* dst_row, const float* gate, void* y,
                          int max_rows, int32_t* status, cudaStream_t stream,
                          int num_sms);

size_t ffn_ws_bytes(int E, int D, int F, int max_rows, int dtype);
// moe_grouped_ffn_variant's answer for valid arguments (1, 2 or 3).
int ffn_variant(int E, int F, int max_rows, int dtype);
moe_status launch_grouped_ffn(int E, int D, int F, int max_rows, int dtype,
                              const void* xp, const int32_t* offsets,
                              const void* w13, const void* w2, void* yp,
                              void* ws, int max_ctas, int32_t* status,
                              cudaStream_t stream, int num_sms);

size_t router_stats_ws_bytes(int T, int E);
moe_status launch_router_stats(int T, int E, int k, int score,
                               const float* logits, const int32_t* topk_idx,
                               float alpha, float* f, float* P,
                               int32_t* counts_routed, float* aux_loss,
                               void* ws, int32_t* status, cudaStream_t stream);
moe_status launch_router_bias_update(int T, int E, int k, float gamma,
                                     const int32_t* counts, float* bias,
                                     cudaStream_t stream);
moe_status launch_dispatch_matrix(int T, int k, int E, int n_src, int n_dst,
                                  const int32_t* topk_idx,
                                  const int32_t* dst_row, int32_t* matrix,
                                  int32_t* status, cudaStream_t stream);
moe_status launch_padded_layout(int T, int k, int E, int capacity,
                                const int32_t* topk_idx,
                                const int32_t* dst_row,
                                const int32_t* offsets,
                                int32_t* dst_row_padded,
                                int32_t* offsets_padded, int32_t* status,
                                cudaStream_t stream);
moe_status launch_pad_fill(int E, int capacity, int D, int dtype,
                           const int32_t* counts, void* buf,
                           cudaStream_t stream, int num_sms);

size_t ffn_bwd_ws_bytes(int F, int max_rows, int dtype);
moe_status launch_grouped_ffn_backward_f32(int E, int D, int F, int max_rows,
                                           const float* xp, const float* dyp,
                                           const int32_t* off,
                                           const float* w13, const float* w2,
                                           float* dxp, float* dw13, float* dw2,
                                           void* ws, cudaStream_t stream);
moe_status launch_grouped_ffn_backward(int E, int D, int F, int max_rows,
                                       const void* xp, const void* dyp,
                                       const int32_t* offsets,
                                       const void* w13, const void* w2,
                                       void* dxp, float* dw13, float* dw2,
                                       void* ws, int32_t* status,
                                       cudaStream_t stream, int num_sms);
moe_status launch_combine_backward(int T, int k, int D, int dtype,
                                   const void* dy, const void* yp,
                                   const int32_t* dst_row, const float* gate,
                                   void* dyp, float* dgate, int max_rows,
                                   int32_t* status, cudaStream_t stream,
                                   int num_sms);
moe_status launch_aligned_layout(int T, int k, int E, int align,
                                 const int32_t* topk_idx,
                                 const int32_t* dst_row,
                                 const int32_t* offsets,
                                 int32_t* dst_row_aligned,
                                 int32_t* offsets_aligned, int32_t* status,
                                 cudaStream_t stream);
moe_status launch_aligned_fill(int E, int D, int dtype, const int32_t* offsets,
                               const int32_t* offsets_aligned, void* buf,
                               cudaStream_t stream);
size_t route_bwd_ws_bytes(int T, int D, int E, int dtype, int num_sms);
bool route_bwd_tensor(int dtype, int E, int D);
bool route_bwd_uses_ws(int dtype, int E, int D, bool dw_r, bool dx);
moe_status launch_route_backward(int T, int D, int E, int k, int score,
                                 int dtype, const void* x, const void* w_r,
                                 const float* logits, const int32_t* topk_idx,
                                 const float* dgate, float* dlogits,
                                 float* dw_r, void* dx, void* ws,
                                 int32_t* status, cudaStream_t stream,
                                 int num_sms);

moe_status launch_sigmoid_key(const float* l, float* out, int n,
                              cudaStream_t stream);
moe_status launch_selftest_wait(int32_t* status, uint64_t limit_ns,
                                cudaStream_t stream);

}  // namespace moe
