"""ctypes binding of libmoe.so (include/moe.h), same entry-point names.

Argument marshalling only: torch tensors become device pointers, the
current CUDA stream becomes the stream argument, and a non-OK status raises
MoeError.  All computation happens in the library's CUDA kernels.  There is
no fallback: if libmoe.so is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_INDEX = 5

MOE_BF16 = 0
MOE_F32 = 1

MOE_SCORE_SOFTMAX_TOPK = 0
MOE_SCORE_SOFTMAX_FULL = 1
MOE_SCORE_SIGMOID_BIAS = 2

SCORE_CODES = {"softmax_topk": MOE_SCORE_SOFTMAX_TOPK,
               "softmax_full": MOE_SCORE_SOFTMAX_FULL,
               "sigmoid_bias": MOE_SCORE_SIGMOID_BIAS}

EXPORTED = ["moe_route_workspace_size", "moe_route_launches", "moe_route",
            "moe_dispatch_layout_workspace_size",
            "moe_dispatch_layout_launches", "moe_dispatch_layout",
            "moe_permute", "moe_grouped_ffn_workspace_size",
            "moe_grouped_ffn_variant",
            "moe_grouped_ffn", "moe_combine", "moe_selftest_bounded_wait",
            "moe_selftest_sigmoid_key", "moe_dispatch_layout_noalloc",
            "moe_router_stats_workspace_size", "moe_router_stats",
            "moe_router_bias_update", "moe_dispatch_matrix",
            "moe_padded_layout", "moe_pad_fill", "moe_aligned_layout",
            "moe_aligned_fill", "moe_combine_backward",
            "moe_permute_backward", "moe_grouped_ffn_backward_workspace_size",
            "moe_grouped_ffn_backward", "moe_route_backward",
            "moe_route_backward_workspace_size", "moe_expert_capacity",
            "moe_status_str", "moe_abi_version"]
ABI_VERSION = 2


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_str(code)} ({code})")


class RouteCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("D", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("score", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("group_score_topk", ctypes.c_int32)]


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64

_SIGS = {
    "moe_route_workspace_size": (_sz, [ctypes.POINTER(RouteCfg)]),
    "moe_route_launches": (_i32, [ctypes.POINTER(RouteCfg)]),
    "moe_route": (_i32, [ctypes.POINTER(RouteCfg), _vp, _vp, _vp, _vp, _vp,
                         _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_dispatch_layout_workspace_size": (_sz, [_i32, _i32, _i32]),
    "moe_dispatch_layout_launches": (_i32, [_i32, _i32, _i32]),
    "moe_dispatch_layout": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   _sz, _vp, _vp]),
    "moe_dispatch_layout_noalloc": (_i32, [_i32, _i32, _i32, _i32, _i32,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp]),
    "moe_permute": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp,
                           _vp]),
    "moe_grouped_ffn_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "moe_grouped_ffn_variant": (_i32, [_i32, _i32, _i32, _i32, _i32]),
    "moe_grouped_ffn": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                               _vp, _vp, _vp, _sz, _i32, _vp, _vp]),
    "moe_combine": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32,
                           _vp, _vp]),
    "moe_expert_capacity": (_i32, [ctypes.c_int64, ctypes.c_int64, _i32, _i32,
                                   _i32]),
    "moe_router_stats_workspace_size": (_sz, [_i32, _i32]),
    "moe_router_stats": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp,
                                ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _sz,
                                _vp, _vp]),
    "moe_router_bias_update": (_i32, [_i32, _i32, _i32, _vp, ctypes.c_float,
                                      _vp, _vp]),
    "moe_dispatch_matrix": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                   _vp, _vp, _vp]),
    "moe_padded_layout": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _vp]),
    "moe_pad_fill": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_aligned_layout": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp]),
    "moe_aligned_fill": (_i32, [_i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "moe_combine_backward": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _i32, _vp, _vp]),
    "moe_permute_backward": (_i32, [_i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                    _i32, _vp, _vp]),
    "moe_grouped_ffn_backward_workspace_size": (_sz, [_i32, _i32, _i32, _i32,
                                                      _i32]),
    "moe_grouped_ffn_backward": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _sz, _vp, _vp]),
    "moe_route_backward": (_i32, [ctypes.POINTER(RouteCfg), _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                  _vp]),
    "moe_route_backward_workspace_size": (_sz, [ctypes.POINTER(RouteCfg)]),
    "moe_selftest_bounded_wait": (_i32, [_vp, _u64, _vp]),
    "moe_selftest_sigmoid_key": (_i32, [_vp, _vp, _i32, _vp]),
    "moe_status_str": (ctypes.c_char_p, [_i32]),
    "moe_abi_version": (_i32, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmoe.so (raises OSError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise OSError(
                f"{path} not found: build it with "
                "`python -m combine_router_gemm_top_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.moe_abi_version() != ABI_VERSION:
            raise OSError("libmoe.so ABI version mismatch; rebuild it")
        _lib = lib
    return _lib


def status_str(code: int) -> str:
    return load().moe_status_str(int(code)).decode()


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(rc, where):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return MOE_BF16
    if dt == torch.float32:
        return MOE_F32
    raise ValueError(f"unsupported dtype {dt}")


def route_cfg(T, D, E, k, dtype, score, n_groups=1, topk_groups=1,
              group_score_topk=0) -> RouteCfg:
    if isinstance(dtype, torch.dtype):
        dtype = dtype_code(dtype)
    if isinstance(score, str):
        score = SCORE_CODES[score]
    return RouteCfg(T, D, E, k, dtype, score, n_groups, topk_groups,
                    group_score_topk)


def moe_route_workspace_size(cfg: RouteCfg) -> int:
    return load().moe_route_workspace_size(ctypes.byref(cfg))


def moe_route_launches(cfg: RouteCfg) -> int:
    return load().moe_route_launches(ctypes.byref(cfg))


def moe_route(cfg, x, w_r, logit_offset, sel_bias, topk_idx, topk_gate,
              logits_out, workspace, status, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().moe_route(ctypes.byref(cfg), _p(x), _p(w_r),
                            _p(logit_offset), _p(sel_bias), _p(topk_idx),
                            _p(topk_gate), _p(logits_out), _p(workspace),
                            nbytes, _p(status), _stream(stream)),
           "moe_route")


def moe_dispatch_layout_workspace_size(T, k, E) -> int:
    return load().moe_dispatch_layout_workspace_size(T, k, E)


def moe_dispatch_layout_launches(T, k, E) -> int:
    return load().moe_dispatch_layout_launches(T, k, E)


def moe_dispatch_layout(T, k, E, R, capacity, topk_idx, expert_counts,
                        expert_offsets, dst_row, src_pair, n_kept, n_dropped,
                        rank_send_counts, rank_send_displs, workspace, status,
                        stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().moe_dispatch_layout(
        T, k, E, R, capacity, _p(topk_idx), _p(expert_counts),
        _p(expert_offsets), _p(dst_row), _p(src_pair), _p(n_kept),
        _p(n_dropped), _p(rank_send_counts), _p(rank_send_displs),
        _p(workspace), nbytes, _p(status), _stream(stream)),
        "moe_dispatch_layout")


def moe_dispatch_layout_noalloc(T, k, E, R, capacity, topk_idx,
                                expert_counts, expert_offsets, dst_row,
                                src_pair, n_kept, n_dropped, rank_send_counts,
                                rank_send_displs, status, stream=None):
    """moe_dispatch_layout without a workspace argument: the library's
    static 1 MiB device scratch is used instead, for callers that cannot
    allocate device memory (see include/moe.h)."""
    _check(load().moe_dispatch_layout_noalloc(
        T, k, E, R, capacity, _p(topk_idx), _p(expert_counts),
        _p(expert_offsets), _p(dst_row), _p(src_pair), _p(n_kept),
        _p(n_dropped), _p(rank_send_counts), _p(rank_send_displs),
        _p(status), _stream(stream)), "moe_dispatch_layout_noalloc")


def _rows(buf, max_rows):
    # rows of a [rows, D] buffer unless the caller names fewer
    return int(buf.shape[0]) if max_rows is None else int(max_rows)


def moe_permute(T, k, D, dtype, x, dst_row, xp, status=None, stream=None,
                max_rows=None):
    _check(load().moe_permute(T, k, D, dtype, _p(x), _p(dst_row), _p(xp),
                              _rows(xp, max_rows), _p(status),
                              _stream(stream)), "moe_permute")


def moe_grouped_ffn_workspace_size(E, D, F, max_rows, dtype) -> int:
    return load().moe_grouped_ffn_workspace_size(E, D, F, max_rows, dtype)


def moe_grouped_ffn_variant(E, D, F, max_rows, dtype) -> int:
    return load().moe_grouped_ffn_variant(E, D, F, max_rows, dtype)


def moe_grouped_ffn(E, D, F, max_rows, dtype, xp, expert_offsets, w13, w2,
                    yp, workspace, status, stream=None, max_ctas=0):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().moe_grouped_ffn(E, D, F, max_rows, dtype, _p(xp),
                                  _p(expert_offsets), _p(w13), _p(w2),
                                  _p(yp), _p(workspace), nbytes,
                                  int(max_ctas), _p(status),
                                  _stream(stream)), "moe_grouped_ffn")


def moe_combine(T, k, D, dtype, yp, dst_row, topk_gate, y, status=None,
                stream=None, max_rows=None):
    _check(load().moe_combine(T, k, D, dtype, _p(yp), _p(dst_row),
                              _p(topk_gate), _p(y), _rows(yp, max_rows),
                              _p(status), _stream(stream)),
           "moe_combine")


def moe_expert_capacity(cf_num, cf_den, T, k, E) -> int:
    """ceil(cf_num / cf_den * k * T / E); -1 for invalid arguments."""
    return load().moe_expert_capacity(int(cf_num), int(cf_den), T, k, E)


def moe_router_stats_workspace_size(T, E) -> int:
    return load().moe_router_stats_workspace_size(T, E)


def moe_router_stats(T, E, k, score, logits, topk_idx, alpha, f, P,
                     counts_routed, aux_loss, workspace, status, stream=None):
    if isinstance(score, str):
        score = SCORE_CODES[score]
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().moe_router_stats(T, E, k, score, _p(logits), _p(topk_idx),
                                   float(alpha), _p(f), _p(P),
                                   _p(counts_routed), _p(aux_loss),
                                   _p(workspace), nbytes, _p(status),
                                   _stream(stream)), "moe_router_stats")


def moe_router_bias_update(T, k, E, counts_routed, gamma, bias, stream=None):
    _check(load().moe_router_bias_update(T, k, E, _p(counts_routed),
                                         float(gamma), _p(bias),
                                         _stream(stream)),
           "moe_router_bias_update")


def moe_dispatch_matrix(T, k, E, n_src, n_dst, topk_idx, dst_row, matrix,
                        status, stream=None):
    _check(load().moe_dispatch_matrix(T, k, E, n_src, n_dst, _p(topk_idx),
                                      _p(dst_row), _p(matrix), _p(status),
                                      _stream(stream)), "moe_dispatch_matrix")


def moe_padded_layout(T, k, E, capacity, topk_idx, dst_row, expert_offsets,
                      dst_row_padded, offsets_padded, status, stream=None):
    _check(load().moe_padded_layout(T, k, E, capacity, _p(topk_idx),
                                    _p(dst_row), _p(expert_offsets),
                                    _p(dst_row_padded), _p(offsets_padded),
                                    _p(status), _stream(stream)),
           "moe_padded_layout")


def moe_pad_fill(E, capacity, D, dtype, expert_counts, buf, stream=None):
    _check(load().moe_pad_fill(E, capacity, D, dtype, _p(expert_counts),
                               _p(buf), _stream(stream)), "moe_pad_fill")


def moe_aligned_layout(T, k, E, align, topk_idx, dst_row, expert_offsets,
                       dst_row_aligned, offsets_aligned, status, stream=None):
    _check(load().moe_aligned_layout(T, k, E, align, _p(topk_idx),
                                     _p(dst_row), _p(expert_offsets),
                                     _p(dst_row_aligned), _p(offsets_aligned),
                                     _p(status), _stream(stream)),
           "moe_aligned_layout")


def moe_aligned_fill(E, D, dtype, expert_offsets, offsets_aligned, buf,
                     stream=None):
    _check(load().moe_aligned_fill(E, D, dtype, _p(expert_offsets),
                                   _p(offsets_aligned), _p(buf),
                                   _stream(stream)), "moe_aligned_fill")


def moe_combine_backward(T, k, D, dtype, dy, yp, dst_row, topk_gate, dyp,
                         dgate, status=None, stream=None, max_rows=None):
    rows = _rows(yp, max_rows if max_rows is not None else
                 min(int(yp.shape[0]), int(dyp.shape[0])))
    _check(load().moe_combine_backward(T, k, D, dtype, _p(dy), _p(yp),
                                       _p(dst_row), _p(topk_gate), _p(dyp),
                                       _p(dgate), rows, _p(status),
                                       _stream(stream)),
           "moe_combine_backward")


def moe_permute_backward(T, k, D, dtype, dxp, dst_row, dx, status=None,
                         stream=None, max_rows=None):
    _check(load().moe_permute_backward(T, k, D, dtype, _p(dxp), _p(dst_row),
                                       _p(dx), _rows(dxp, max_rows),
                                       _p(status), _stream(stream)),
           "moe_permute_backward")


def moe_grouped_ffn_backward_workspace_size(E, D, F, max_rows, dtype) -> int:
    return load().moe_grouped_ffn_backward_workspace_size(E, D, F, max_rows,
                                                          dtype)


def moe_grouped_ffn_backward(E, D, F, max_rows, dtype, xp, dyp,
                             expert_offsets, w13, w2, dxp, dw13, dw2,
                             workspace, status, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().moe_grouped_ffn_backward(
        E, D, F, max_rows, dtype, _p(xp), _p(dyp), _p(expert_offsets),
        _p(w13), _p(w2), _p(dxp), _p(dw13), _p(dw2), _p(workspace), nbytes,
        _p(status), _stream(stream)), "moe_grouped_ffn_backward")


def moe_route_backward_workspace_size(cfg) -> int:
    return load().moe_route_backward_workspace_size(ctypes.byref(cfg))


def moe_route_backward(cfg, x, w_r, logits, topk_idx, dgate, dlogits, dw_r,
                       dx, workspace, status, stream=None):
    nbytes = 0 if workspace is None else \
        workspace.numel() * workspace.element_size()
    _check(load().moe_route_backward(ctypes.byref(cfg), _p(x), _p(w_r),
                                     _p(logits), _p(topk_idx), _p(dgate),
                                     _p(dlogits), _p(dw_r), _p(dx),
                                     _p(workspace), nbytes, _p(status),
                                     _stream(stream)),
           "moe_route_backward")


def moe_selftest_bounded_wait(status, limit_ns, stream=None):
    _check(load().moe_selftest_bounded_wait(_p(status), int(limit_ns),
                                            _stream(stream)),
           "moe_selftest_bounded_wait")


def moe_selftest_sigmoid_key(l, out, stream=None):
    _check(load().moe_selftest_sigmoid_key(_p(l), _p(out), l.numel(),
                                           _stream(stream)),
           "moe_selftest_sigmoid_key")
