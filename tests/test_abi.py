"""CPU checks of the C ABI: libmoe.so builds and loads, exports every
function include/moe.h declares, and rejects bad arguments on the host
(MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED) before launching anything.  No call
here reaches a kernel, so these run without a GPU."""
import ctypes
import os
import re

import pytest

from combine_router_gemm_top_b300 import _lib as L
from combine_router_gemm_top_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    B.build(verbose=False)
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(",
                                 text)))


def test_every_csrc_file_is_built_or_watched():
    # an edit to any file under csrc/ must rebuild the library
    csrc = os.path.join(ROOT, "combine_router_gemm_top_b300", "csrc")
    files = sorted(f for f in os.listdir(csrc)
                   if os.path.isfile(os.path.join(csrc, f)))
    assert files
    watched = set(B.SOURCES) | set(B.headers())
    assert [f for f in files if f not in watched] == []
    assert "umma_ffn.cuh" in B.headers()


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch_layout", "moe_permute",
              "moe_grouped_ffn", "moe_combine"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert sorted(L.EXPORTED) == names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.moe_abi_version() == L.ABI_VERSION


def test_status_strings(lib):
    assert L.status_str(0) == "MOE_OK"
    assert L.status_str(4) == "MOE_ERR_TIMEOUT"
    assert L.status_str(99) == "MOE_ERR_UNKNOWN"


FAKE = 1 << 20   # a non-null, 256-byte aligned address that is never touched


def test_route_rejects_bad_configs(lib):
    good = L.route_cfg(128, 256, 8, 2, L.MOE_BF16, L.MOE_SCORE_SOFTMAX_TOPK)
    assert L.moe_route_workspace_size(good) > 0
    bad = [L.route_cfg(128, 256, 8, 9, L.MOE_BF16, 0),       # k > E
           L.route_cfg(128, 256, 300, 2, L.MOE_BF16, 0),     # E > 256
           L.route_cfg(128, 250, 8, 2, L.MOE_BF16, 0),       # row not 16 B
           L.route_cfg(128, 256, 8, 2, 7, 0),                # dtype
           L.route_cfg(128, 256, 8, 2, L.MOE_BF16, 5),       # score
           L.route_cfg(128, 256, 12, 2, L.MOE_BF16, 2, 5, 1, 1),   # groups
           L.route_cfg(128, 256, 16, 8, L.MOE_BF16, 2, 4, 1, 2)]   # k > kept
    for cfg in bad:
        assert L.moe_route_workspace_size(cfg) == 0
        rc = lib.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, FAKE,
                           FAKE, None, FAKE, 1 << 30, None, None)
        assert rc == L.MOE_ERR_INVALID
    # null pointers and misalignment
    rc = lib.moe_route(ctypes.byref(good), None, FAKE, None, None, FAKE, FAKE,
                       None, FAKE, 1 << 30, None, None)
    assert rc == L.MOE_ERR_INVALID
    rc = lib.moe_route(ctypes.byref(good), FAKE + 16, FAKE, None, None, FAKE,
                       FAKE, None, FAKE, 1 << 30, None, None)
    assert rc == L.MOE_ERR_INVALID
    # workspace too small
    rc = lib.moe_route(ctypes.byref(good), FAKE, FAKE, None, None, FAKE, FAKE,
                       None, FAKE, 4, None, None)
    assert rc == L.MOE_ERR_INVALID


def test_layout_rejects_bad_sizes(lib):
    assert lib.moe_dispatch_layout_workspace_size(10, 2, 8) > 0
    assert lib.moe_dispatch_layout_workspace_size(10, 33, 64) == 0
    args = [FAKE] * 9 + [FAKE, 1 << 30, None, None]
    assert lib.moe_dispatch_layout(10, 2, 8, 3, 0, *args) == L.MOE_ERR_INVALID
    assert lib.moe_dispatch_layout(10, 2, 8, 0, 0, *args) == L.MOE_ERR_INVALID
    assert lib.moe_dispatch_layout(10, 2, 2048, 8, 0, *args) == \
        L.MOE_ERR_INVALID
    assert lib.moe_dispatch_layout(1 << 30, 4, 8, 8, 0, *args) == \
        L.MOE_ERR_INVALID                              # T*k overflows int32
    small = [FAKE] * 9 + [FAKE, 4, None, None]
    assert lib.moe_dispatch_layout(10, 2, 8, 4, 0, *small) == \
        L.MOE_ERR_INVALID                              # workspace too small
    nul = [FAKE] * 9 + [None, 1 << 30, None, None]
    assert lib.moe_dispatch_layout(10, 2, 8, 4, 0, *nul) == L.MOE_ERR_INVALID


def test_route_launches(lib):
    # one kernel up to 32 experts: in bf16 (the MMA router) for E <= 8, a
    # padded W_r of <= 96 KiB, or T <= 16 tokens per SM; in fp32 for a
    # padded W_r of <= 96 KiB (in shared memory); the bf16 router GEMM alone
    # when it selects in its epilogue (one K split, softmax, no groups,
    # k <= 2, E <= 64); else GEMM + select
    for E, D, dt, n in [(8, 4096, L.MOE_BF16, 1), (32, 1024, L.MOE_BF16, 1),
                        (32, 4096, L.MOE_BF16, 1), (8, 65536, L.MOE_BF16, 1),
                        (33, 64, L.MOE_BF16, 1), (64, 4096, L.MOE_BF16, 2),
                        (256, 4096, L.MOE_BF16, 2),
                        (8, 3072, L.MOE_F32, 1), (8, 4096, L.MOE_F32, 2),
                        (32, 1024, L.MOE_F32, 2)]:
        cfg = L.route_cfg(2048, D, E, 2, dt, 0)
        assert lib.moe_route_launches(ctypes.byref(cfg)) == n, (E, D, dt)
    # above one 16-token tile per SM, bf16 W_r over 96 KiB with more than 8
    # experts goes back to the GEMM (148 SMs without a device)
    for T, E, D, n in [(16384, 32, 4096, 1), (16384, 16, 4096, 1),
                       (16384, 8, 4096, 1), (16384, 32, 1024, 1)]:
        cfg = L.route_cfg(T, D, E, 2, L.MOE_BF16, 0)
        assert lib.moe_route_launches(ctypes.byref(cfg)) == n, (T, E, D)
    # the fused GEMM: one K split at the Switch-like shape; not with the
    # sigmoid score, groups, k > 2, E > 64 or several K splits
    for (T, D, E, k, score, groups), n in [
            ((16384, 1024, 64, 1, 1, (1, 1, 0)), 1),
            ((16384, 1024, 40, 2, 0, (1, 1, 0)), 1),
            ((16384, 1024, 65, 1, 0, (1, 1, 0)), 2),
            ((16384, 1024, 64, 1, 2, (1, 1, 0)), 2),
            ((16384, 1024, 64, 2, 0, (4, 2, 2)), 2),
            ((16384, 1024, 64, 3, 0, (1, 1, 0)), 2),
            ((16384, 1024, 144, 1, 0, (1, 1, 0)), 2),
            ((2048, 1024, 64, 1, 1, (1, 1, 0)), 2)]:
        cfg = L.route_cfg(T, D, E, k, L.MOE_BF16, score, *groups)
        assert lib.moe_route_launches(ctypes.byref(cfg)) == n, (T, D, E, k)
    assert lib.moe_route_launches(ctypes.byref(
        L.route_cfg(0, 4096, 8, 2, L.MOE_BF16, 0))) == 0
    assert lib.moe_route_launches(ctypes.byref(
        L.route_cfg(128, 256, 8, 9, L.MOE_BF16, 0))) == 0


def test_layout_launches(lib):
    # one block up to 16384 pairs and 256 experts, else three kernels
    assert lib.moe_dispatch_layout_launches(2048, 2, 8) == 1
    assert lib.moe_dispatch_layout_launches(16384, 1, 64) == 1
    assert lib.moe_dispatch_layout_launches(4096, 8, 128) == 3
    assert lib.moe_dispatch_layout_launches(1000, 2, 300) == 3
    assert lib.moe_dispatch_layout_launches(0, 2, 300) == 1
    assert lib.moe_dispatch_layout_launches(16, 33, 8) == 0
    assert lib.moe_dispatch_layout_launches(16, 2, 2000) == 0


def test_grouped_ffn_variant(lib):
    # 1: fp32 FMA, one block per row (F <= 12288); 4: fp32 FMA, up then
    # down; 2: one SM per 128-row tile; 3: SM pairs, taken for F % 256 == 0,
    # E <= 256 and max_rows >= 384 E; 0: rejected or empty
    bf, f32 = L.MOE_BF16, L.MOE_F32
    for args, v in [((8, 4096, 14336, 4096, bf), 3),     # Mixtral-like
                    ((8, 4096, 14336, 3071, bf), 2),
                    ((8, 4096, 14336, 3072, bf), 3),
                    ((8, 4096, 14208, 8192, bf), 2),     # F % 256 = 128
                    ((256, 7168, 2048, 32768, bf), 2),   # DeepSeek-like
                    ((256, 7168, 2048, 98304, bf), 3),
                    ((256, 256, 256, 384 * 256, bf), 3),
                    ((256, 256, 256, 384 * 256 - 1, bf), 2),
                    ((257, 256, 256, 1 << 20, bf), 2),   # E > 256
                    ((64, 1024, 4096, 16384, bf), 2),    # Switch-like
                    ((8, 64, 128, 4096, f32), 1),
                    ((8, 64, 12288, 4096, f32), 1),
                    ((8, 64, 12289, 4096, f32), 4),
                    ((8, 4096, 14336, 0, bf), 0),
                    ((8, 4000, 14336, 4096, bf), 0),     # D % 64 != 0
                    ((0, 4096, 14336, 4096, bf), 0)]:
        assert lib.moe_grouped_ffn_variant(*args) == v, args


def test_permute_combine_reject(lib):
    R = 20   # rows of the expert-contiguous buffer
    assert lib.moe_permute(10, 2, 12, L.MOE_BF16, FAKE, FAKE, FAKE, R, None,
                           None) == L.MOE_ERR_INVALID   # 24-byte rows
    assert lib.moe_permute(10, 2, 16, L.MOE_BF16, None, FAKE, FAKE, R, None,
                           None) == L.MOE_ERR_INVALID
    assert lib.moe_permute(10, 2, 16, L.MOE_BF16, FAKE + 8, FAKE, FAKE, R,
                           None, None) == L.MOE_ERR_INVALID
    assert lib.moe_permute(10, 2, 16, L.MOE_BF16, FAKE, FAKE, FAKE, -1,
                           None, None) == L.MOE_ERR_INVALID   # max_rows < 0
    assert lib.moe_combine(10, 40, 16, L.MOE_BF16, FAKE, FAKE, FAKE, FAKE, R,
                           None, None) == L.MOE_ERR_INVALID   # k > 32
    assert lib.moe_combine(10, 2, 16, 3, FAKE, FAKE, FAKE, FAKE, R, None,
                           None) == L.MOE_ERR_INVALID
    assert lib.moe_combine(10, 2, 16, L.MOE_BF16, FAKE, FAKE, FAKE, FAKE, -5,
                           None, None) == L.MOE_ERR_INVALID
    assert lib.moe_combine_backward(10, 2, 16, L.MOE_BF16, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, FAKE, -1, None, None) == \
        L.MOE_ERR_INVALID
    assert lib.moe_permute_backward(10, 2, 16, L.MOE_BF16, FAKE, FAKE, FAKE,
                                    -1, None, None) == L.MOE_ERR_INVALID
    # nothing to do is not an error
    assert lib.moe_permute(0, 2, 16, L.MOE_BF16, None, None, None, 0, None,
                           None) == L.MOE_OK


def test_expert_capacity_matches_the_oracle(lib):
    # the library's integer evaluation of ceil(CF * k * T / E) against the
    # oracle's rational one over a grid of factors and shapes
    import oracle.moe_oracle as O
    from fractions import Fraction
    for cf in ("0.5", "1", "1.0", "1.1", "1.25", "1.5", "2", "3.75", "0.01"):
        f = Fraction(cf)
        for T, k, E in [(256, 2, 8), (16384, 1, 64), (100, 2, 8), (10, 1, 4),
                        (1, 1, 256), (0, 2, 8), (65536, 8, 128), (7, 3, 5)]:
            got = lib.moe_expert_capacity(f.numerator, f.denominator, T, k, E)
            assert got == O.expert_capacity(cf, T, k, E), (cf, T, k, E)
    assert lib.moe_expert_capacity(5, 4, 256, 2, 8) == 80
    assert lib.moe_expert_capacity(1, 1, 16384, 1, 64) == 256
    assert lib.moe_expert_capacity(-1, 1, 10, 1, 4) == -1
    assert lib.moe_expert_capacity(1, 0, 10, 1, 4) == -1
    assert lib.moe_expert_capacity(1, 1, 10, 0, 4) == -1
    assert lib.moe_expert_capacity(1, 1, 10, 1, 0) == -1
    assert lib.moe_expert_capacity(1 << 40, 1, 1 << 30, 32, 1) == -1   # > INT32_MAX
    assert lib.moe_expert_capacity((1 << 62), (1 << 62), 1 << 30, 1, 1) == 1 << 30


def test_grouped_ffn_reject(lib):
    ok_ws = 1 << 40
    assert lib.moe_grouped_ffn(8, 100, 256, 64, L.MOE_BF16, FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, ok_ws, 0, None, None) == \
        L.MOE_ERR_UNSUPPORTED                          # D % 64
    assert lib.moe_grouped_ffn(8, 128, 200, 64, L.MOE_BF16, FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, ok_ws, 0, None, None) == \
        L.MOE_ERR_UNSUPPORTED                          # F % 128
    assert lib.moe_grouped_ffn(8, 128, 256, 64, L.MOE_BF16, FAKE + 16, FAKE,
                               FAKE, FAKE, FAKE, FAKE, ok_ws, 0, None, None) == \
        L.MOE_ERR_INVALID                              # TMA base alignment
    assert lib.moe_grouped_ffn(8, 128, 256, 64, L.MOE_BF16, FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, 16, 0, None, None) == \
        L.MOE_ERR_INVALID                              # workspace too small
    assert lib.moe_grouped_ffn(8, 128, 256, 64, L.MOE_BF16, FAKE, None, FAKE,
                               FAKE, FAKE, FAKE, ok_ws, 0, None, None) == \
        L.MOE_ERR_INVALID
    # H [max_rows, F], then one counter per row block (ceil(64/128) + E) and
    # the SM-pair launch's tile ticket
    assert lib.moe_grouped_ffn_workspace_size(8, 128, 256, 64, L.MOE_BF16) == \
        64 * 256 * 2 + (1 + 8 + 1) * 4
    assert lib.moe_grouped_ffn_workspace_size(8, 128, 256, 64, L.MOE_F32) == \
        64 * 256 * 4


def test_route_backward_reject(lib):
    # bf16 with E and D multiples of 64: dx and dw_r run on the tensor cores
    # through the dL2 workspace, so dx alone needs a workspace
    tc = L.route_cfg(128, 128, 64, 2, L.MOE_BF16, L.MOE_SCORE_SOFTMAX_TOPK)
    need = L.moe_route_backward_workspace_size(tc)
    assert need >= 128 * 2 * 64 * 2            # dL2 [T, 2E] bf16
    def call(cfg, dw_r, dx, ws, ws_bytes, x=FAKE):
        return lib.moe_route_backward(ctypes.byref(cfg), x, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, dw_r, dx, ws, ws_bytes,
                                      None, None)
    assert call(tc, None, FAKE, None, 0) == L.MOE_ERR_INVALID
    assert call(tc, None, FAKE, FAKE, need - 1) == L.MOE_ERR_INVALID
    assert call(tc, None, FAKE + 8, FAKE, need) == L.MOE_ERR_INVALID
    assert call(tc, FAKE, None, FAKE, need, x=FAKE + 8) == L.MOE_ERR_INVALID
    assert call(tc, FAKE, None, FAKE + 8, need) == L.MOE_ERR_INVALID
    # missing inputs
    assert call(tc, FAKE, None, FAKE, need, x=None) == L.MOE_ERR_INVALID
    bad = L.route_cfg(128, 128, 64, 65, L.MOE_BF16, 0)
    assert L.moe_route_backward_workspace_size(bad) == 0
    assert call(bad, None, None, None, 0) == L.MOE_ERR_INVALID


def test_selftests_reject_null(lib):
    assert lib.moe_selftest_bounded_wait(None, 10, None) == L.MOE_ERR_INVALID
    assert lib.moe_selftest_sigmoid_key(None, None, 5, None) == \
        L.MOE_ERR_INVALID
