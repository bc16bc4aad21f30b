// C-ABI entry points of libmoe.so (declared in include/moe.h): argument
// validation, workspace sizing, tensor-map encoding and launch.  Every
// error the host can see is reported here before anything is launched.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

int g_sms[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return kNumSMs;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        n <= 0)
      n = kNumSMs;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool valid_dtype(int32_t d) { return d == MOE_BF16 || d == MOE_F32; }

}  // namespace

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t cols,
                       int64_t rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool route_cfg_ok(const moe_route_cfg* c) {
  if (c == nullptr) return false;
  if (c->T < 0 || c->D <= 0 || c->E < 1 || c->E > 256) return false;
  if (c->k < 1 || c->k > c->E || c->k > 32) return false;
  if (!valid_dtype(c->dtype)) return false;
  if (c->score < MOE_SCORE_SOFTMAX_TOPK || c->score > MOE_SCORE_SIGMOID_BIAS)
    return false;
  if (c->n_groups < 1 || c->n_groups > 32 || c->E % c->n_groups != 0)
    return false;
  if (c->n_groups > 1) {
    const int gs = c->E / c->n_groups;
    if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return false;
    if (c->group_score_topk < 1 || c->group_score_topk > gs) return false;
    if (c->topk_groups * gs < c->k) return false;
  }
  if ((static_cast<int64_t>(c->D) * dtype_bytes(c->dtype)) % 16 != 0)
    return false;
  if (static_cast<int64_t>(c->T) * c->E * 8 > INT32_MAX) return false;
  return true;
}

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_str(int32_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_INDEX: return "MOE_ERR_INDEX";
    default: return "MOE_ERR_UNKNOWN";
  }
}

size_t moe_route_workspace_size(const moe_route_cfg* cfg) {
  if (!route_cfg_ok(cfg)) return 0;
  const size_t b = plan_route(*cfg, num_sms()).ws_bytes;
  return b > 0 ? b : 16;
}

int32_t moe_route_launches(const moe_route_cfg* cfg) {
  if (!route_cfg_ok(cfg) || cfg->T == 0) return 0;
  const int sms = num_sms();
  return route_single_kernel(*cfg, sms) || route_fused_gemm(*cfg, sms) ? 1 : 2;
}

moe_status moe_route(const moe_route_cfg* cfg, const void* x, const void* w_r,
                     const float* logit_offset, const float* sel_bias,
                     int32_t* topk_idx, float* topk_gate, float* logits_out,
                     void* workspace, size_t workspace_bytes, int32_t* status,
                     moe_stream_t stream) {
  if (!route_cfg_ok(cfg)) return MOE_ERR_INVALID;
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || w_r == nullptr || topk_idx == nullptr ||
      topk_gate == nullptr || workspace == nullptr)
    return MOE_ERR_INVALID;
  const size_t a = cfg->dtype == MOE_BF16 ? 256 : 16;
  if (!aligned(x, a) || !aligned(w_r, a) || !aligned(workspace, 16))
    return MOE_ERR_INVALID;
  const int sms = num_sms();
  if (workspace_bytes < plan_route(*cfg, sms).ws_bytes) return MOE_ERR_INVALID;
  return launch_route(*cfg, x, w_r, logit_offset, sel_bias, topk_idx,
                      topk_gate, logits_out, workspace, status,
                      reinterpret_cast<cudaStream_t>(stream), sms);
}

size_t moe_dispatch_layout_workspace_size(int32_t T, int32_t k, int32_t E) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > kLayoutMaxE) return 0;
  return layout_ws_bytes(static_cast<int64_t>(T) * k, E);
}

int32_t moe_dispatch_layout_launches(int32_t T, int32_t k, int32_t E) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > kLayoutMaxE) return 0;
  return layout_launches(static_cast<int64_t>(T) * k, E);
}

moe_status moe_dispatch_layout(int32_t T, int32_t k, int32_t E, int32_t R,
                               int32_t capacity, const int32_t* topk_idx,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* dst_row, int32_t* src_pair,
                               int32_t* n_kept, int32_t* n_dropped,
                               int32_t* rank_send_counts,
                               int32_t* rank_send_displs, void* workspace,
                               size_t workspace_bytes, int32_t* status,
                               moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > kLayoutMaxE) return MOE_ERR_INVALID;
  if (R < 1 || R > E || E % R != 0) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(T) * k > INT32_MAX) return MOE_ERR_INVALID;
  if (expert_counts == nullptr || expert_offsets == nullptr ||
      n_kept == nullptr || n_dropped == nullptr ||
      rank_send_counts == nullptr || rank_send_displs == nullptr ||
      workspace == nullptr)
    return MOE_ERR_INVALID;
  if (T > 0 && (topk_idx == nullptr || dst_row == nullptr || src_pair == nullptr))
    return MOE_ERR_INVALID;
  if (!aligned(workspace, 16)) return MOE_ERR_INVALID;
  if (workspace_bytes < layout_ws_bytes(static_cast<int64_t>(T) * k, E))
    return MOE_ERR_INVALID;
  return launch_layout(T, k, E, R, capacity, topk_idx, expert_counts,
                       expert_offsets, dst_row, src_pair, n_kept, n_dropped,
                       rank_send_counts, rank_send_displs, workspace, status,
                       reinterpret_cast<cudaStream_t>(stream));
}

static bool rows_ok(int32_t T, int32_t k, int32_t D, int32_t dtype) {
  if (T < 0 || k < 1 || k > 32 || D <= 0 || !valid_dtype(dtype)) return false;
  if ((static_cast<int64_t>(D) * dtype_bytes(dtype)) % 16 != 0) return false;
  if (static_cast<int64_t>(T) * k > INT32_MAX) return false;
  return true;
}

moe_status moe_permute(int32_t T, int32_t k, int32_t D, int32_t dtype,
                       const void* x, const int32_t* dst_row, void* xp,
                       int32_t max_rows, int32_t* status,
                       moe_stream_t stream) {
  if (!rows_ok(T, k, D, dtype) || max_rows < 0) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if (x == nullptr || dst_row == nullptr || (xp == nullptr && max_rows > 0))
    return MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(xp, 16)) return MOE_ERR_INVALID;
  return launch_permute(T, k, D, dtype, x, dst_row, xp, max_rows, status,
                        reinterpret_cast<cudaStream_t>(stream), num_sms());
}

moe_status moe_combine(int32_t T, int32_t k, int32_t D, int32_t dtype,
                       const void* yp, const int32_t* dst_row,
                       const float* topk_gate, void* y, int32_t max_rows,
                       int32_t* status, moe_stream_t stream) {
  if (!rows_ok(T, k, D, dtype) || max_rows < 0) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if ((yp == nullptr && max_rows > 0) || dst_row == nullptr ||
      topk_gate == nullptr || y == nullptr)
    return MOE_ERR_INVALID;
  if (!aligned(yp, 16) || !aligned(y, 16)) return MOE_ERR_INVALID;
  return launch_combine(T, k, D, dtype, yp, dst_row, topk_gate, y, max_rows,
                        status, reinterpret_cast<cudaStream_t>(stream),
                        num_sms());
}

int32_t moe_expert_capacity(int64_t cf_num, int64_t cf_den, int32_t T,
                            int32_t k, int32_t E) {
  if (cf_num < 0 || cf_den <= 0 || T < 0 || k < 1 || E < 1) return -1;
  // ceil(cf_num * k * T / (cf_den * E)); every product fits in 128 bits
  const unsigned __int128 num = static_cast<unsigned __int128>(cf_num) *
                                static_cast<uint64_t>(k) *
                                static_cast<uint64_t>(T);
  const unsigned __int128 den = static_cast<unsigned __int128>(cf_den) *
                                static_cast<uint64_t>(E);
  const unsigned __int128 c = (num + den - 1) / den;
  if (c > static_cast<unsigned __int128>(INT32_MAX)) return -1;
  return static_cast<int32_t>(c);
}

size_t moe_grouped_ffn_workspace_size(int32_t E, int32_t D, int32_t F,
                                      int32_t max_rows, int32_t dtype) {
  if (E < 1 || D <= 0 || F <= 0 || max_rows < 0 || !valid_dtype(dtype)) return 0;
  const size_t b = ffn_ws_bytes(E, D, F, max_rows, dtype);
  return b > 0 ? b : 16;
}

// Shape and dtype checks of moe_grouped_ffn (pointers aside).
static moe_status ffn_shape_status(int32_t E, int32_t D, int32_t F,
                                   int32_t max_rows, int32_t dtype) {
  if (E < 1 || D <= 0 || F <= 0 || max_rows < 0 || !valid_dtype(dtype))
    return MOE_ERR_INVALID;
  if (dtype == MOE_BF16) {
    if (D % 64 != 0 || F % 128 != 0 || E > kMaxGroupsApi)
      return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * 2 * F > INT32_MAX ||
        static_cast<int64_t>(E) * D > INT32_MAX)
      return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

int32_t moe_grouped_ffn_variant(int32_t E, int32_t D, int32_t F,
                                int32_t max_rows, int32_t dtype) {
  if (ffn_shape_status(E, D, F, max_rows, dtype) != MOE_OK || max_rows == 0)
    return 0;
  return ffn_variant(E, F, max_rows, dtype);
}

moe_status moe_grouped_ffn(int32_t E, int32_t D, int32_t F, int32_t max_rows,
                           int32_t dtype, const void* xp,
                           const int32_t* expert_offsets, const void* w13,
                           const void* w2, void* yp, void* workspace,
                           size_t workspace_bytes, int32_t max_ctas,
                           int32_t* status, moe_stream_t stream) {
  if (E < 1 || D <= 0 || F <= 0 || max_rows < 0 || !valid_dtype(dtype))
    return MOE_ERR_INVALID;
  if (max_rows == 0) return MOE_OK;
  if (xp == nullptr || expert_offsets == nullptr || w13 == nullptr ||
      w2 == nullptr || yp == nullptr || workspace == nullptr)
    return MOE_ERR_INVALID;
  if (workspace_bytes < ffn_ws_bytes(E, D, F, max_rows, dtype))
    return MOE_ERR_INVALID;
  const moe_status shape = ffn_shape_status(E, D, F, max_rows, dtype);
  if (shape != MOE_OK) return shape;
  if (dtype == MOE_BF16) {
    if (!aligned(xp, 256) || !aligned(w13, 256) || !aligned(w2, 256) ||
        !aligned(yp, 16) || !aligned(workspace, 256))
      return MOE_ERR_INVALID;
  } else {
    if (!aligned(xp, 16) || !aligned(yp, 16) || !aligned(workspace, 16))
      return MOE_ERR_INVALID;
  }
  return launch_grouped_ffn(E, D, F, max_rows, dtype, xp, expert_offsets, w13,
                            w2, yp, workspace, max_ctas, status,
                            reinterpret_cast<cudaStream_t>(stream), num_sms());
}

size_t moe_router_stats_workspace_size(int32_t T, int32_t E) {
  if (T < 0 || E < 1 || E > 256) return 0;
  return router_stats_ws_bytes(T, E);
}

moe_status moe_router_stats(int32_t T, int32_t E, int32_t k, int32_t score,
                            const float* logits, const int32_t* topk_idx,
                            float alpha, float* f, float* P,
                            int32_t* counts_routed, float* aux_loss,
                            void* workspace, size_t workspace_bytes,
                            int32_t* status, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > E || k > 32)
    return MOE_ERR_INVALID;
  if (score < MOE_SCORE_SOFTMAX_TOPK || score > MOE_SCORE_SIGMOID_BIAS)
    return MOE_ERR_INVALID;
  if (static_cast<int64_t>(T) * E > INT32_MAX) return MOE_ERR_INVALID;
  if (f == nullptr || P == nullptr || aux_loss == nullptr ||
      workspace == nullptr)
    return MOE_ERR_INVALID;
  if (T > 0 && (logits == nullptr || topk_idx == nullptr))
    return MOE_ERR_INVALID;
  if (!aligned(workspace, 16) || workspace_bytes < router_stats_ws_bytes(T, E))
    return MOE_ERR_INVALID;
  return launch_router_stats(T, E, k, score, logits, topk_idx, alpha, f, P,
                             counts_routed, aux_loss, workspace, status,
                             reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_router_bias_update(int32_t T, int32_t k, int32_t E,
                                  const int32_t* counts_routed, float gamma,
                                  float* bias, moe_stream_t stream) {
  if (T < 0 || k < 1 || E < 1 || counts_routed == nullptr || bias == nullptr)
    return MOE_ERR_INVALID;
  return launch_router_bias_update(T, E, k, gamma, counts_routed, bias,
                                   reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch_matrix(int32_t T, int32_t k, int32_t E, int32_t n_src,
                               int32_t n_dst, const int32_t* topk_idx,
                               const int32_t* dst_row, int32_t* matrix,
                               int32_t* status, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || n_src < 1 || n_dst < 1 ||
      n_dst > 4096 || E % n_dst != 0)
    return MOE_ERR_INVALID;
  if (T % n_src != 0 || static_cast<int64_t>(T) * k > INT32_MAX)
    return MOE_ERR_INVALID;
  if (static_cast<int64_t>(n_src) * n_dst > INT32_MAX || n_src > 65535)
    return MOE_ERR_INVALID;
  if (matrix == nullptr || (T > 0 && topk_idx == nullptr))
    return MOE_ERR_INVALID;
  return launch_dispatch_matrix(T, k, E, n_src, n_dst, topk_idx, dst_row,
                                matrix, status,
                                reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_padded_layout(int32_t T, int32_t k, int32_t E, int32_t capacity,
                             const int32_t* topk_idx, const int32_t* dst_row,
                             const int32_t* expert_offsets,
                             int32_t* dst_row_padded, int32_t* offsets_padded,
                             int32_t* status, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || capacity < 1) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(E) * capacity > INT32_MAX ||
      static_cast<int64_t>(T) * k > INT32_MAX)
    return MOE_ERR_INVALID;
  if (expert_offsets == nullptr || offsets_padded == nullptr)
    return MOE_ERR_INVALID;
  if (T > 0 && (topk_idx == nullptr || dst_row == nullptr ||
                dst_row_padded == nullptr))
    return MOE_ERR_INVALID;
  return launch_padded_layout(T, k, E, capacity, topk_idx, dst_row,
                              expert_offsets, dst_row_padded, offsets_padded,
                              status, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_pad_fill(int32_t E, int32_t capacity, int32_t D, int32_t dtype,
                        const int32_t* expert_counts, void* buf,
                        moe_stream_t stream) {
  if (E < 1 || capacity < 1 || !rows_ok(1, 1, D, dtype)) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(E) * capacity > INT32_MAX) return MOE_ERR_INVALID;
  if (expert_counts == nullptr || buf == nullptr || !aligned(buf, 16))
    return MOE_ERR_INVALID;
  return launch_pad_fill(E, capacity, D, dtype, expert_counts, buf,
                         reinterpret_cast<cudaStream_t>(stream), num_sms());
}

moe_status moe_aligned_layout(int32_t T, int32_t k, int32_t E, int32_t align,
                              const int32_t* topk_idx, const int32_t* dst_row,
                              const int32_t* expert_offsets,
                              int32_t* dst_row_aligned,
                              int32_t* offsets_aligned, int32_t* status,
                              moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > kLayoutMaxE || align < 1 ||
      align > 1024)
    return MOE_ERR_INVALID;
  if (static_cast<int64_t>(T) * k + static_cast<int64_t>(align - 1) * E >
      INT32_MAX)
    return MOE_ERR_INVALID;
  if (expert_offsets == nullptr || offsets_aligned == nullptr)
    return MOE_ERR_INVALID;
  if (T > 0 && (topk_idx == nullptr || dst_row == nullptr ||
                dst_row_aligned == nullptr))
    return MOE_ERR_INVALID;
  return launch_aligned_layout(T, k, E, align, topk_idx, dst_row,
                               expert_offsets, dst_row_aligned,
                               offsets_aligned, status,
                               reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_aligned_fill(int32_t E, int32_t D, int32_t dtype,
                            const int32_t* expert_offsets,
                            const int32_t* offsets_aligned, void* buf,
                            moe_stream_t stream) {
  if (E < 1 || !rows_ok(1, 1, D, dtype)) return MOE_ERR_INVALID;
  if (expert_offsets == nullptr || offsets_aligned == nullptr ||
      buf == nullptr || !aligned(buf, 16))
    return MOE_ERR_INVALID;
  return launch_aligned_fill(E, D, dtype, expert_offsets, offsets_aligned,
                             buf, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_combine_backward(int32_t T, int32_t k, int32_t D, int32_t dtype,
                                const void* dy, const void* yp,
                                const int32_t* dst_row, const float* topk_gate,
                                void* dyp, float* dgate, int32_t max_rows,
                                int32_t* status, moe_stream_t stream) {
  if (!rows_ok(T, k, D, dtype) || max_rows < 0) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if (dy == nullptr || dst_row == nullptr || topk_gate == nullptr ||
      dgate == nullptr ||
      ((yp == nullptr || dyp == nullptr) && max_rows > 0))
    return MOE_ERR_INVALID;
  if (!aligned(dy, 16) || !aligned(yp, 16) || !aligned(dyp, 16))
    return MOE_ERR_INVALID;
  return launch_combine_backward(T, k, D, dtype, dy, yp, dst_row, topk_gate,
                                 dyp, dgate, max_rows, status,
                                 reinterpret_cast<cudaStream_t>(stream),
                                 num_sms());
}

moe_status moe_permute_backward(int32_t T, int32_t k, int32_t D, int32_t dtype,
                                const void* dxp, const int32_t* dst_row,
                                void* dx, int32_t max_rows, int32_t* status,
                                moe_stream_t stream) {
  if (!rows_ok(T, k, D, dtype) || max_rows < 0) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if ((dxp == nullptr && max_rows > 0) || dst_row == nullptr || dx == nullptr)
    return MOE_ERR_INVALID;
  if (!aligned(dxp, 16) || !aligned(dx, 16)) return MOE_ERR_INVALID;
  return launch_combine(T, k, D, dtype, dxp, dst_row, nullptr, dx, max_rows,
                        status, reinterpret_cast<cudaStream_t>(stream),
                        num_sms());
}

size_t moe_grouped_ffn_backward_workspace_size(int32_t E, int32_t D, int32_t F,
                                               int32_t max_rows,
                                               int32_t dtype) {
  if (E < 1 || D <= 0 || F <= 0 || max_rows < 0 || !valid_dtype(dtype))
    return 0;
  const size_t b = ffn_bwd_ws_bytes(F, max_rows, dtype);
  return b > 0 ? b : 16;
}

moe_status moe_grouped_ffn_backward(
    int32_t E, int32_t D, int32_t F, int32_t max_rows, int32_t dtype,
    const void* xp, const void* dyp, const int32_t* expert_offsets,
    const void* w13, const void* w2, void* dxp, float* dw13, float* dw2,
    void* workspace, size_t workspace_bytes, int32_t* status,
    moe_stream_t stream) {
  if (E < 1 || D <= 0 || F <= 0 || max_rows < 0 || !valid_dtype(dtype))
    return MOE_ERR_INVALID;
  if (dtype == MOE_F32) {
    if (xp == nullptr || dyp == nullptr || expert_offsets == nullptr ||
        w13 == nullptr || w2 == nullptr || dxp == nullptr ||
        dw13 == nullptr || dw2 == nullptr || workspace == nullptr)
      return MOE_ERR_INVALID;
    if (!aligned(workspace, 16) ||
        workspace_bytes < ffn_bwd_ws_bytes(F, max_rows, dtype))
      return MOE_ERR_INVALID;
    if (static_cast<int64_t>(E) * 2 * F * D > INT32_MAX * 64LL)
      return MOE_ERR_UNSUPPORTED;
    if (max_rows == 0) return MOE_OK;
    return launch_grouped_ffn_backward_f32(
        E, D, F, max_rows, static_cast<const float*>(xp),
        static_cast<const float*>(dyp), expert_offsets,
        static_cast<const float*>(w13), static_cast<const float*>(w2),
        static_cast<float*>(dxp), dw13, dw2, workspace,
        reinterpret_cast<cudaStream_t>(stream));
  }
  if (D % 128 != 0 || F % 128 != 0 || E > kMaxGroupsApi)
    return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * 2 * F > INT32_MAX ||
      static_cast<int64_t>(E) * D > INT32_MAX)
    return MOE_ERR_UNSUPPORTED;
  if (xp == nullptr || dyp == nullptr || expert_offsets == nullptr ||
      w13 == nullptr || w2 == nullptr || dxp == nullptr || dw13 == nullptr ||
      dw2 == nullptr || workspace == nullptr)
    return MOE_ERR_INVALID;
  if (!aligned(xp, 256) || !aligned(dyp, 256) || !aligned(w13, 256) ||
      !aligned(w2, 256) || !aligned(workspace, 256) || !aligned(dxp, 16) ||
      !aligned(dw13, 16) || !aligned(dw2, 16))
    return MOE_ERR_INVALID;
  if (workspace_bytes < ffn_bwd_ws_bytes(F, max_rows, dtype))
    return MOE_ERR_INVALID;
  return launch_grouped_ffn_backward(E, D, F, max_rows, xp, dyp,
                                     expert_offsets, w13, w2, dxp, dw13, dw2,
                                     workspace, status,
                                     reinterpret_cast<cudaStream_t>(stream),
                                     num_sms());
}

size_t moe_route_backward_workspace_size(const moe_route_cfg* cfg) {
  if (!route_cfg_ok(cfg)) return 0;
  const size_t b =
      route_bwd_ws_bytes(cfg->T, cfg->D, cfg->E, cfg->dtype, num_sms());
  return b > 0 ? b : 16;
}

moe_status moe_route_backward(const moe_route_cfg* cfg, const void* x,
                              const void* w_r, const float* logits,
                              const int32_t* topk_idx, const float* dgate,
                              float* dlogits, float* dw_r, void* dx,
                              void* workspace, size_t workspace_bytes,
                              int32_t* status, moe_stream_t stream) {
  if (!route_cfg_ok(cfg)) return MOE_ERR_INVALID;
  if (cfg->T == 0) return MOE_OK;
  if (logits == nullptr || topk_idx == nullptr || dgate == nullptr ||
      dlogits == nullptr)
    return MOE_ERR_INVALID;
  if (dw_r != nullptr && x == nullptr) return MOE_ERR_INVALID;
  if (dx != nullptr && w_r == nullptr) return MOE_ERR_INVALID;
  if (route_bwd_tensor(cfg->dtype, cfg->E, cfg->D) &&
      ((dw_r != nullptr && !aligned(x, 16)) ||
       (dx != nullptr && (!aligned(dx, 16) || !aligned(w_r, 16)))))
    return MOE_ERR_INVALID;
  const int sms = num_sms();
  const size_t need =
      route_bwd_ws_bytes(cfg->T, cfg->D, cfg->E, cfg->dtype, sms);
  if (route_bwd_uses_ws(cfg->dtype, cfg->E, cfg->D, dw_r != nullptr,
                        dx != nullptr) &&
      need > 0 &&
      (workspace == nullptr || workspace_bytes < need ||
       !aligned(workspace, 16)))
    return MOE_ERR_INVALID;
  return launch_route_backward(cfg->T, cfg->D, cfg->E, cfg->k, cfg->score,
                               cfg->dtype, x, w_r, logits, topk_idx, dgate,
                               dlogits, dw_r, dx, workspace, status,
                               reinterpret_cast<cudaStream_t>(stream), sms);
}

moe_status moe_selftest_bounded_wait(int32_t* status, uint64_t limit_ns,
                                     moe_stream_t stream) {
  if (status == nullptr) return MOE_ERR_INVALID;
  return launch_selftest_wait(status, limit_ns,
                              reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_selftest_sigmoid_key(const float* l, float* out, int32_t n,
                                    moe_stream_t stream) {
  if (n < 0) return MOE_ERR_INVALID;
  if (n > 0 && (l == nullptr || out == nullptr)) return MOE_ERR_INVALID;
  return launch_sigmoid_key(l, out, n, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
