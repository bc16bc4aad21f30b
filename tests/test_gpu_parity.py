"""GPU parity: every step of the CUDA path, called through the C ABI,
against the CPU oracle on the same seeded inputs.

Bars (written into each check):
  * integers (top-k ids, counts, offsets, dst_row, src_pair, rank counts):
    bit-exact; routing ids are checked on the logits the kernel used
    (logits_out), so both sides take the selection on the same fp32 values;
  * gates: |g - g_ref| <= 2e-6;
  * router logits: |l - l_ref| <= 2^-16 * sum_d |x_d w_d| + 1e-6 (fp32
    accumulation against the float64 dot product);
  * layer / expert outputs: max|y - y_ref| / max|y_ref| <= 1e-5 (fp32) or
    <= 1e-2 (bf16).
"""
import math

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from combine_router_gemm_top_b300 import _lib as L
from combine_router_gemm_top_b300 import workloads as W
from combine_router_gemm_top_b300.layer import MoELayer, expert_capacity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def i64(t):
    return t.detach().to("cpu", torch.int64).numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return np.abs(got - ref).max() / (den if den > 0 else 1.0)


def tol_for(dtype):
    return 1e-5 if dtype == torch.float32 else 1e-2


# ------------------------------------------------------------ bounded wait
def test_bounded_wait_reports_timeout():
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_selftest_bounded_wait(st, 2_000_000)      # 2 ms
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0


# ------------------------------------------------------------ layout
def run_layout(idx, E, R, cap):
    T, k = idx.shape
    P = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(counts=torch.full((E,), -7, **i32),
               offsets=torch.full((E + 1,), -7, **i32),
               dst_row=torch.full((max(P, 1),), -7, **i32),
               src_pair=torch.full((max(P, 1),), -7, **i32),
               n_kept=torch.full((1,), -7, **i32),
               n_dropped=torch.full((1,), -7, **i32),
               rc=torch.full((R,), -7, **i32), rd=torch.full((R,), -7, **i32))
    ws = torch.empty(max(L.moe_dispatch_layout_workspace_size(T, k, E), 16),
                     dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, **i32)
    d_idx = torch.as_tensor(np.ascontiguousarray(idx), dtype=torch.int32,
                            device=DEV)
    L.moe_dispatch_layout(T, k, E, R, cap, d_idx, out["counts"],
                          out["offsets"], out["dst_row"], out["src_pair"],
                          out["n_kept"], out["n_dropped"], out["rc"],
                          out["rd"], ws, st)
    torch.cuda.synchronize()
    out["status"] = st
    return {key: i64(v) for key, v in out.items()}


def check_layout(g, ref, P):
    assert g["counts"].tolist() == ref["counts"].tolist()
    assert g["offsets"].tolist() == ref["offsets"].tolist()
    assert g["dst_row"][:P].tolist() == ref["dst_row"].tolist()
    n = ref["n_kept"]
    assert int(g["n_kept"][0]) == n and int(g["n_dropped"][0]) == P - n
    assert g["src_pair"][:n].tolist() == ref["src_pair"].tolist()
    assert g["rc"].tolist() == ref["rank_send_counts"].tolist()
    assert g["rd"].tolist() == ref["rank_send_displs"].tolist()


def _idx(kind, T, k, E, seed):
    rng = np.random.default_rng(seed)
    if kind == "distinct":
        return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    if kind == "dup":
        return rng.integers(0, E, size=(T, k)).astype(np.int32)
    if kind == "one":
        return np.full((T, k), E - 1, dtype=np.int32)
    if kind == "skew":     # Zipf-like: many pairs on the first experts
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        return rng.choice(E, size=(T, k), p=p / p.sum()).astype(np.int32)
    raise ValueError(kind)


LAYOUT_CASES = [
    (1, 1, 1, 1, 0, "dup"), (1, 2, 8, 4, 0, "distinct"),
    (31, 2, 8, 4, 0, "distinct"), (33, 2, 8, 4, 1, "distinct"),
    (256, 2, 8, 4, 80, "distinct"), (2048, 2, 8, 8, 0, "distinct"),
    (2048 * 3 + 5, 8, 128, 8, 0, "skew"), (16384, 1, 64, 16, 256, "skew"),
    (5000, 4, 64, 16, 0, "one"), (5000, 4, 64, 16, 100, "one"),
    (3001, 8, 256, 8, 100, "dup"), (4096, 8, 256, 8, 0, "distinct"),
    (1500, 3, 1024, 32, 2, "dup"), (65536, 8, 128, 8, 0, "distinct"),
    # more than 256 chunks of 2048 pairs: the scan takes several batches
    (70000, 8, 64, 8, 0, "dup"),
    # either side of the one-block layout (<= 16384 pairs, <= 256 experts)
    (2048, 8, 256, 8, 30, "skew"), (2049, 8, 64, 8, 0, "dup"),
    (2000, 2, 260, 4, 0, "dup"), (4096, 8, 256, 8, 60, "skew"),
]


@pytest.mark.parametrize("T,k,E,R,cap,kind", LAYOUT_CASES)
def test_layout_bit_exact(T, k, E, R, cap, kind):
    idx = _idx(kind, T, k, E, seed=T + E)
    g = run_layout(idx, E, R, cap)
    ref = O.dispatch_layout(idx, E, R, cap if cap > 0 else None)
    check_layout(g, ref, T * k)
    assert int(g["status"][0]) == 0


@pytest.mark.parametrize("E,R,cap", [(8, 4, 0), (300, 4, 5)])
def test_layout_empty_batch(E, R, cap):
    # T = 0: every count, offset, rank count and displacement is 0 (the
    # one-block path for E = 8, the three-launch path for E = 300)
    idx = np.zeros((0, 2), dtype=np.int32)
    g = run_layout(idx, E, R, cap)
    ref = O.dispatch_layout(idx, E, R, cap or None)
    check_layout(g, ref, 0)
    assert int(g["status"][0]) == 0


def test_layout_page_worked_example():
    idx = np.array([[0, 2], [1, 3], [0, 1], [2, 3]], dtype=np.int32)
    g = run_layout(idx, 4, 2, 0)
    assert g["rc"].tolist() == [4, 4]
    assert g["src_pair"][:8].tolist() == [0, 4, 2, 5, 1, 6, 3, 7]


def test_layout_out_of_range_ids_are_dropped_and_reported():
    T, k, E = 700, 2, 16
    idx = _idx("dup", T, k, E, seed=5)
    idx[3, 1] = -1
    idx[100, 0] = E
    idx[650, 1] = 1 << 20
    g = run_layout(idx, E, 4, 0)
    assert int(g["status"][0]) == L.MOE_ERR_INDEX
    # reference: invalid pairs go to an extra expert E that is then ignored
    fixed = np.where((idx < 0) | (idx >= E), E, idx)
    ref = O.dispatch_layout(fixed, E + 1, 1, None)
    bad = ((idx < 0) | (idx >= E)).reshape(-1)
    dst = ref["dst_row"].copy()
    dst[bad] = -1
    assert g["dst_row"][:T * k].tolist() == dst.tolist()
    assert g["offsets"].tolist() == ref["offsets"][:E + 1].tolist()
    assert int(g["n_dropped"][0]) == int(bad.sum())


def test_layout_deterministic():
    idx = _idx("skew", 9000, 8, 128, seed=1)
    a = run_layout(idx, 128, 8, 300)
    b = run_layout(idx, 128, 8, 300)
    for key in a:
        assert (a[key] == b[key]).all()


# ------------------------------------------------------------ route
def make_route_inputs(T, D, E, dtype, seed, w_std=None, offset=None,
                      bias=None):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((T, D), generator=g).to(dtype)
    std = w_std if w_std is not None else 1.0 / math.sqrt(D)
    w = (torch.randn((E, D), generator=g) * std).to(dtype)
    off = None
    if offset is not None:
        off = (offset * torch.log(1.0 / torch.arange(1, E + 1,
                                                     dtype=torch.float64))
               ).float()
    b = None
    if bias is not None:
        b = (torch.rand(E, generator=g) * 2 - 1) * bias
    return x, w, off, b


def run_route(x, w, off, b, k, score, groups=(1, 1, 0)):
    T, D = x.shape
    E = w.shape[0]
    cfg = L.route_cfg(T, D, E, k, x.dtype, score, *groups)
    ws = torch.empty(max(L.moe_route_workspace_size(cfg), 16),
                     dtype=torch.uint8, device=DEV)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    gate = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dx, dw = x.to(DEV), w.to(DEV)
    doff = off.to(DEV) if off is not None else None
    db = b.to(DEV) if b is not None else None
    L.moe_route(cfg, dx, dw, doff, db, idx, gate, logits, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return i64(idx), f64(gate), logits.cpu().numpy()


def check_route(x, w, off, b, k, score, groups, idx, gate, logits):
    x64, w64 = f64(x), f64(w)
    ref_l = O.router_logits(x64, w64, None if off is None else off.numpy())
    bound = 2.0 ** -16 * (np.abs(x64) @ np.abs(w64).T) + 1e-6
    assert np.isfinite(logits).all()
    assert (np.abs(logits.astype(np.float64) - ref_l) <= bound).all()
    ridx, rgate = O.route_from_logits(
        logits, k, score, None if b is None else b.numpy(), *groups)
    assert (idx == ridx).all()
    assert np.abs(gate - rgate).max() <= 2e-6


ROUTE_CASES = [
    # T, D, E, k, dtype, score, groups, w_std, offset, bias
    (256, 64, 8, 2, torch.float32, "softmax_topk", (1, 1, 0), 0.02, None, None),
    (300, 256, 8, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (129, 64, 16, 4, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (1000, 512, 64, 1, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    (777, 1024, 256, 8, torch.bfloat16, "sigmoid_bias", (8, 4, 2), None, None, 0.1),
    (257, 200, 40, 3, torch.bfloat16, "sigmoid_bias", (4, 2, 3), None, None, 0.3),
    (64, 128, 4, 4, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (1, 64, 8, 1, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (513, 96, 24, 5, torch.float32, "sigmoid_bias", (3, 2, 2), None, None, 0.05),
    # more than 32 experts in fp32: the FMA router GEMM, then the select kernel
    (300, 64, 40, 3, torch.float32, "softmax_topk", (1, 1, 0), 0.02, None, None),
    # 32 experts exactly: the one-kernel router at its widest
    (700, 1024, 32, 4, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    # one-kernel router: bf16 over 24 chunks per warp (two load batches);
    # fp32 W_r exactly at its 96 KiB shared-memory limit; 5 experts padded
    # to 8 zero rows with a ragged chunk count (D = 520); 12 experts (16
    # rows) with the group limit
    (150, 6144, 8, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (150, 3072, 8, 2, torch.float32, "softmax_topk", (1, 1, 0), 0.02, None, None),
    (333, 520, 5, 2, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.0, None),
    (200, 320, 12, 3, torch.bfloat16, "sigmoid_bias", (4, 2, 2), None, None, 0.1),
    # few experts, long rows: bf16 stays on the one-kernel router (32
    # chunks per warp, several load batches); fp32 W_r over the 96 KiB
    # shared-memory limit takes the FMA router GEMM, then the select kernel
    (257, 8192, 8, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (130, 4096, 8, 2, torch.float32, "softmax_topk", (1, 1, 0), 0.02, None, None),
    # group scores over more than 8 keys (the warp-round path)
    (333, 128, 64, 6, torch.bfloat16, "sigmoid_bias", (4, 2, 12), None, None, 0.2),
    (300, 128, 96, 8, torch.bfloat16, "softmax_topk", (6, 3, 16), None, None, None),
    # 32 groups of 8, every lane scoring one group
    (400, 256, 256, 8, torch.bfloat16, "sigmoid_bias", (32, 6, 2), None, None, 0.1),
    # E not a multiple of 32, groups straddling lanes
    (211, 128, 200, 7, torch.bfloat16, "sigmoid_bias", (8, 3, 5), None, None, 0.1),
    # many row blocks, one K split, ragged last row block
    (10000, 256, 128, 8, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (9500, 128, 64, 1, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    (12000, 64, 8, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (20000, 128, 200, 5, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (10000, 128, 64, 9, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    # more row blocks than SMs, unevenly: the GEMM runs as two K halves
    (20000, 512, 64, 4, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (10000, 128, 64, 4, torch.bfloat16, "softmax_topk", (4, 2, 2), None, None, None),
    # one-kernel router at and above one block per SM, odd T (bf16: token
    # tiles of 14 and 16 rows with a ragged last tile; fp32: more than 8 warps
    # per SM): 8, 16 and 32 expert rows, every score mode
    (2049, 4096, 8, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (1999, 256, 32, 4, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    (3001, 520, 12, 3, torch.bfloat16, "sigmoid_bias", (4, 2, 2), None, None, 0.1),
    (1501, 96, 24, 5, torch.float32, "sigmoid_bias", (3, 2, 2), None, None, 0.05),
    (1301, 64, 16, 4, torch.float32, "softmax_topk", (1, 1, 0), 0.02, None, None),
    # bf16, 16 and 32 experts with W_r over 96 KiB: the MMA router while T
    # fits one 16-token tile per SM, the router GEMM (16 columns) above that
    (2300, 4096, 32, 4, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    (3000, 4096, 16, 4, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    # the router GEMM selecting in its epilogue (one K split, softmax, k <=
    # 2, E <= 64): the Switch-like shape, 60 experts (a ragged last column
    # chunk), 40 and 33 experts; then 100 experts, past it
    (16384, 1024, 64, 1, torch.bfloat16, "softmax_full", (1, 1, 0), None, 1.5, None),
    (10000, 256, 60, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
    (12000, 512, 40, 2, torch.bfloat16, "softmax_full", (1, 1, 0), None, None, None),
    (10500, 128, 33, 1, torch.bfloat16, "softmax_topk", (1, 1, 0), None, 0.5, None),
    (10000, 256, 100, 2, torch.bfloat16, "softmax_topk", (1, 1, 0), None, None, None),
]


@pytest.mark.parametrize("case", ROUTE_CASES)
def test_route_parity(case):
    T, D, E, k, dt, score, groups, w_std, offset, bias = case
    x, w, off, b = make_route_inputs(T, D, E, dt, seed=T * 7 + E, w_std=w_std,
                                     offset=offset, bias=bias)
    idx, gate, logits = run_route(x, w, off, b, k, score, groups)
    check_route(x, w, off, b, k, score, groups, idx, gate, logits)


@pytest.mark.parametrize("E,D,dt", [(8, 4096, torch.bfloat16),
                                    (32, 256, torch.bfloat16),
                                    (16, 64, torch.float32)])
def test_route_logits_independent_of_batch_size(E, D, dt):
    # a token's logits are formed by its own warp in a fixed order, so they
    # are the same bits whatever the call's T (one block or many per SM) and
    # wherever the token sits in the batch
    T = 4001
    x, w, _, _ = make_route_inputs(T, D, E, dt, seed=E + D)
    _, _, big = run_route(x, w, None, None, 2, "softmax_topk")
    _, _, small = run_route(x[:100], w, None, None, 2, "softmax_topk")
    assert np.array_equal(big[:100].view(np.int32), small.view(np.int32))
    _, _, tail = run_route(x[-37:], w, None, None, 2, "softmax_topk")
    assert np.array_equal(big[-37:].view(np.int32), tail.view(np.int32))


@pytest.mark.parametrize("T,E,k", [(512, 16, 4), (10240, 16, 4),
                                   (10240, 64, 2), (10240, 64, 1)])
def test_route_ties_go_to_lower_index(T, E, k):
    # D = E and w_r = identity: logits equal x exactly (small integers in
    # bf16), so many experts tie; the lower index must win every tie (64
    # experts at T = 10240: the router GEMM selecting in its epilogue)
    rng = np.random.default_rng(3)
    xl = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    x = torch.tensor(xl).to(torch.bfloat16)
    w = torch.eye(E).to(torch.bfloat16)
    idx, gate, logits = run_route(x, w, None, None, k, "softmax_topk")
    assert (logits == xl).all()
    ridx, rgate = O.route_from_logits(xl, k, "softmax_topk")
    assert (idx == ridx).all()
    assert np.abs(gate - rgate).max() <= 2e-6


@pytest.mark.parametrize("groups", [(8, 3, 2), (4, 2, 8), (2, 1, 12)])
def test_route_group_ties_go_to_lower_index(groups):
    # integer logits: equal keys and equal group scores everywhere; the lower
    # group and the lower expert must win every tie
    T, E, k = 640, 32, 5
    rng = np.random.default_rng(11)
    xl = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    x = torch.tensor(xl).to(torch.bfloat16)
    w = torch.eye(E).to(torch.bfloat16)
    idx, gate, logits = run_route(x, w, None, None, k, "softmax_topk", groups)
    assert (logits == xl).all()
    ridx, rgate = O.route_from_logits(xl, k, "softmax_topk", None, *groups)
    assert (idx == ridx).all()
    assert np.abs(gate - rgate).max() <= 2e-6


@pytest.mark.parametrize("E,groups,k", [(256, (8, 4, 2), 8), (64, (1, 1, 0), 6),
                                         (32, (4, 2, 3), 4), (256, (8, 3, 8), 8)])
def test_sigmoid_route_near_ties(E, groups, k):
    # sigmoid keys that differ by a few fp32 ulp (logits on a fine grid, bias
    # steps of 2^-23): the approximate keys cannot order these experts, so
    # most of them must go through the exact evaluation (several rounds of
    # 32); ids must still equal the oracle's definitional selection, bit for
    # bit, on the logits the kernel used
    T, D = 96, 64
    g = torch.Generator().manual_seed(E + k)
    # x . w = one-hot rows of w pick logits from a fine grid around 0.3
    x = torch.zeros((T, D))
    x[:, 0] = 1.0
    w = torch.zeros((E, D))
    w[:, 0] = 0.3 + torch.randint(-40, 40, (E,), generator=g).float() * 2.0 ** -22
    for t in range(T):
        x[t, 1 + t % (D - 1)] = 2.0 ** -20 * (t % 7)
    w[:, 1:] = torch.randint(-3, 4, (E, D - 1), generator=g).float()
    b = torch.randint(-4, 5, (E,), generator=g).float() * 2.0 ** -23
    idx, gate, logits = run_route(x.float(), w.float(), None, b, k,
                                  "sigmoid_bias", groups)
    ridx, rgate = O.route_from_logits(logits, k, "sigmoid_bias", b.numpy(),
                                      *groups)
    assert (idx == ridx).all()
    assert np.abs(gate - rgate).max() <= 2e-6


@pytest.mark.parametrize("E,groups,k,dt", [
    (64, (8, 4, 2), 8, torch.float32), (256, (8, 4, 2), 8, torch.bfloat16),
    (64, (1, 1, 0), 6, torch.bfloat16), (32, (4, 2, 2), 4, torch.float32)])
def test_sigmoid_route_paired_ties(E, groups, k, dt):
    # experts in pairs with the same router row, their biases 0 or 1 ulp of
    # a key apart: logits spread widely, so few experts are near the k-th
    # key, but every pair is a near-tie (an exact tie in a third of them)
    # that the approximate keys cannot order; ids must equal the oracle's
    # definitional selection bit for bit, ties to the lower index
    T, D = 300, 64
    g = torch.Generator().manual_seed(E * 7 + k)
    x = torch.randn((T, D), generator=g)
    w = torch.randn((E // 2, D), generator=g) * D ** -0.5
    w = w.repeat_interleave(2, dim=0)
    b = (torch.rand(E // 2, generator=g) * 0.2 - 0.1).repeat_interleave(2)
    step = torch.randint(-1, 2, (E // 2,), generator=g).float()
    b[1::2] = b[1::2] + step * 2.0 ** -24
    x = x.to(dt).float()
    w = w.to(dt).float()
    idx, gate, logits = run_route(x.to(dt), w.to(dt), None, b, k,
                                  "sigmoid_bias", groups)
    assert (logits[:, 0::2] == logits[:, 1::2]).all()   # paired logits
    ridx, rgate = O.route_from_logits(logits, k, "sigmoid_bias", b.numpy(),
                                      *groups)
    assert (idx == ridx).all()
    assert np.abs(gate - rgate).max() <= 2e-6


def test_sigmoid_key_bit_exact():
    # the selection score is an integer decision's input: the device's
    # fp32(sigmoid(l)) must equal the oracle's float64 sigmoid rounded once
    # (itself pinned against scipy's expit and a 50-digit evaluation).  A
    # difference is allowed only where the float64 value sits within 2^-44
    # (relative) of the midpoint between two fp32 values, where two float64
    # evaluations may round either way; none is expected.
    l = np.concatenate([np.linspace(-95, 95, 1 << 20),
                        np.random.default_rng(8).standard_normal(1 << 18) * 6,
                        [0.0, -0.0, 17.9, 18.0, 87.0, -87.0, 88.0, -88.0,
                         103.0, -103.0, 1e-30, -1e-30]]).astype(np.float32)
    dl = torch.tensor(l, device=DEV)
    out = torch.empty_like(dl)
    L.moe_selftest_sigmoid_key(dl, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = O.sigmoid_f32(l)
    diff = got.view(np.uint32) != ref.view(np.uint32)
    if diff.any():
        s64 = O.sigmoid_f64(l[diff])
        lo = np.minimum(got[diff], ref[diff]).astype(np.float64)
        hi = np.maximum(got[diff], ref[diff]).astype(np.float64)
        adjacent = np.nextafter(lo.astype(np.float32), np.float32(2)) == \
            hi.astype(np.float32)
        near_mid = np.abs(s64 - (lo + hi) / 2) <= 2.0 ** -44 * s64
        assert (adjacent & near_mid).all(), l[diff][~(adjacent & near_mid)][:8]
    assert diff.sum() <= 2


# ------------------------------------------------------------ permute/combine
@pytest.mark.parametrize("T,k,E,D,dt,cap", [
    (1, 1, 4, 8, torch.bfloat16, 0), (37, 2, 8, 64, torch.bfloat16, 0),
    (300, 8, 16, 520, torch.bfloat16, 30), (129, 2, 8, 64, torch.float32, 20),
    (2048, 8, 128, 4096, torch.bfloat16, 0),
    # rows cut into 2 segments of 192 vectors, and into 4 with drops
    (777, 2, 8, 3072, torch.bfloat16, 0), (500, 2, 8, 2048, torch.float32, 40),
    # top-1 at capacity, most tokens dropped whole: their rows are not read
    (4000, 1, 64, 1024, torch.bfloat16, 30),
    # more tokens than the grid's 148 x 64 warps, so warps take a
    # second token, with rows of 16 vectors (fewer than a warp's lanes), of
    # 129 vectors (one past a step of 128) and of 10 vectors; k = 1 and 4
    # take the general combine loop
    (12000, 1, 64, 128, torch.bfloat16, 100),
    (12000, 1, 8, 516, torch.float32, 0),
    (10000, 4, 16, 40, torch.float32, 1500)])
def test_permute_combine_parity(T, k, E, D, dt, cap):
    idx = _idx("distinct", T, k, E, seed=D)
    lay = O.dispatch_layout(idx, E, 1, cap if cap > 0 else None)
    dst = torch.tensor(lay["dst_row"], dtype=torch.int32, device=DEV)
    g = torch.Generator().manual_seed(T)
    x = torch.randn((T, D), generator=g).to(dt)
    gates = torch.rand((T, k), generator=g)
    gates = (gates / gates.sum(1, keepdim=True)).float()
    P = T * k
    xp = torch.full((P, D), float("nan"), dtype=dt, device=DEV)
    dx = x.to(DEV)
    L.moe_permute(T, k, D, L.dtype_code(dt), dx, dst, xp)
    torch.cuda.synchronize()
    n = lay["n_kept"]
    ref_xp = O.permute(f64(x), lay["src_pair"], k)
    assert (f64(xp[:n]) == ref_xp).all()            # a copy: bit-exact
    assert torch.isnan(xp[n:].float()).all()        # untouched past n_kept
    yp = (torch.randn((P, D), generator=g)).to(dt).to(DEV)
    y = torch.full((T, D), float("nan"), dtype=dt, device=DEV)
    L.moe_combine(T, k, D, L.dtype_code(dt), yp, dst, gates.to(DEV), y)
    torch.cuda.synchronize()
    ref_y = O.combine(f64(yp), lay["dst_row"], f64(gates), T, k)
    assert rel_err(f64(y), ref_y) <= tol_for(dt)
    # fp32 accumulation then one rounding: each element within one output
    # ulp plus the fp32 accumulation error
    if dt == torch.bfloat16:
        assert (np.abs(f64(y) - ref_y) <= np.abs(ref_y) * 2 ** -8 + 1e-6).all()


# ------------------------------------------------------------ grouped FFN
def run_ffn(xp, counts, w13, w2, F, sentinel=True, max_ctas=0):
    E = len(counts)
    D = xp.shape[1]
    max_rows = xp.shape[0]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d_off = torch.tensor(off, device=DEV)
    dt = xp.dtype
    yp = torch.full((max_rows, D), float("nan") if sentinel else 0.0,
                    dtype=dt, device=DEV)
    ws = torch.empty(max(L.moe_grouped_ffn_workspace_size(
        E, D, F, max_rows, L.dtype_code(dt)), 16), dtype=torch.uint8,
        device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_grouped_ffn(E, D, F, max_rows, L.dtype_code(dt), xp.to(DEV), d_off,
                      w13.to(DEV), w2.to(DEV), yp, ws, st, max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert st.item() == 0
    return yp, off


FFN_CASES = [
    # E, D, F, counts, dtype
    (4, 128, 256, [0, 1, 200, 129], torch.bfloat16),
    (6, 256, 256, [255, 256, 257, 16, 17, 513], torch.bfloat16),
    (3, 256, 128, [128, 256, 5], torch.bfloat16),
    (1, 512, 384, [300], torch.bfloat16),
    (5, 192, 256, [7, 0, 0, 130, 64], torch.bfloat16),
    (8, 1024, 512, [100, 300, 0, 17, 128, 129, 255, 1], torch.bfloat16),
    (8, 64, 128, [10, 50, 0, 3, 128, 70, 1, 250], torch.float32),
    # fp32 with D and F not multiples of a warp's 32 lanes (one block per
    # row), and F past the shared-memory row buffer (up, then down)
    (3, 36, 100, [5, 40, 33], torch.float32),
    (2, 40, 12300, [7, 20], torch.float32),
    # tails of every swapped MMA width (16..112) and the 112/113 switch to
    # the normal tile; D = 320 leaves a down-projection tile half outside D
    (8, 256, 256, [16, 33, 112, 113, 128 + 48, 256 + 97, 240, 2],
     torch.bfloat16),
    (7, 320, 128, [40, 170, 3, 81, 128 + 65, 0, 97], torch.bfloat16),
    (2, 768, 384, [1, 64], torch.bfloat16),
    # more tiles than SMs in both projections (21 row blocks, D = 2048),
    # with swapped tails, and fewer down tiles than SMs (16 row blocks)
    (4, 2048, 128, [600, 700, 513, 640], torch.bfloat16),
    (3, 2048, 128, [600, 700, 513], torch.bfloat16),
    # long down-projection contractions (32 and 16 K blocks) over few tiles,
    # swapped and normal
    (4, 512, 2048, [300, 40, 0, 129], torch.bfloat16),
    (1, 256, 1024, [1000], torch.bfloat16),
    # short tails (1..49 rows) after one or more full row blocks of the same
    # expert, next to other experts' rows and, for the last expert, next to
    # the unused rows at the end of the allocation
    (7, 256, 256, [128 + 47, 256 + 48, 128 + 49, 384 + 16, 128 + 33, 0,
                   128 + 1], torch.bfloat16),
    (3, 320, 384, [256 + 32, 48, 128 + 48], torch.bfloat16),
]


@pytest.mark.parametrize("case", FFN_CASES)
def test_grouped_ffn_parity(case):
    E, D, F, counts, dt = case
    n = sum(counts)
    max_rows = n + 37
    g = torch.Generator().manual_seed(E * 1000 + D)
    xp = torch.randn((max_rows, D), generator=g).to(dt)
    std = 1.0 / math.sqrt(D)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * std).to(dt)
    w2 = (torch.randn((E, D, F), generator=g) * std).to(dt)
    yp, off = run_ffn(xp, counts, w13, w2, F)
    ref = O.grouped_ffn(f64(xp)[:n], off, f64(w13), f64(w2))
    got = f64(yp[:n])
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= tol_for(dt)
    assert torch.isnan(yp[n:].float()).all()


PAIR_FFN_CASES = [
    # E, D, F, counts: experts averaging >= 384 rows run on SM pairs with
    # 256-row blocks.  Tails of 1..64 rows run swapped; longer remainders
    # are a block whose rows past the expert's are computed, not stored.
    (2, 256, 512, [256 + 1, 512 + 64]),
    (3, 320, 256, [256 + 65, 128, 512 + 16]),      # D = 320: half-outside
    (4, 256, 256, [40, 0, 700, 256 + 44]),         # a tail-only expert
    (2, 512, 512, [512, 256]),                     # full blocks only
    (1, 256, 1024, [1000]),                        # 16 K blocks down
    (8, 1024, 512, [100, 300, 0, 17, 128, 129, 255, 1]),
    (1, 64, 256, [400]),                           # one K block up
    (16, 128, 256, [300, 511, 512, 513, 320, 257, 575, 576, 577, 0, 64,
                    700, 310, 450, 290, 333]),
]


def pair_ffn_inputs(E, D, F, counts, seed):
    n = sum(counts)
    max_rows = max(n + 37, 384 * E)
    assert L.moe_grouped_ffn_variant(E, D, F, max_rows,
                                     L.dtype_code(torch.bfloat16)) == 3
    g = torch.Generator().manual_seed(seed)
    xp = torch.randn((max_rows, D), generator=g).to(torch.bfloat16)
    std = 1.0 / math.sqrt(D)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * std).to(torch.bfloat16)
    w2 = (torch.randn((E, D, F), generator=g) * std).to(torch.bfloat16)
    return n, xp, w13, w2


@pytest.mark.parametrize("case", PAIR_FFN_CASES)
def test_grouped_ffn_pairs_parity(case):
    E, D, F, counts = case
    n, xp, w13, w2 = pair_ffn_inputs(E, D, F, counts, seed=E * 77 + D)
    yp, off = run_ffn(xp, counts, w13, w2, F)
    ref = O.grouped_ffn(f64(xp)[:n], off, f64(w13), f64(w2))
    got = f64(yp[:n])
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= tol_for(torch.bfloat16)
    assert torch.isnan(yp[n:].float()).all()


@pytest.mark.parametrize("ctas", [2, 8, 37])
def test_grouped_ffn_pairs_on_few_ctas(ctas):
    # the pair launch on a grid of a few clusters (an odd request rounds
    # down to whole pairs): same bits as on every SM
    E, D, F, counts = 3, 512, 512, [600, 40, 513]
    n, xp, w13, w2 = pair_ffn_inputs(E, D, F, counts, seed=93)
    yp, off = run_ffn(xp, counts, w13, w2, F, max_ctas=ctas)
    ref = O.grouped_ffn(f64(xp)[:n], off, f64(w13), f64(w2))
    assert rel_err(f64(yp[:n]), ref) <= 1e-2
    full, _ = run_ffn(xp, counts, w13, w2, F)
    assert torch.equal(yp[:n], full[:n])


@pytest.mark.parametrize("ctas", [1, 8, 37])
def test_grouped_ffn_on_few_ctas(ctas):
    # the persistent launch on a grid far below the SM count: every CTA walks
    # many up tiles and then down tiles that wait for up tiles other CTAs
    # hold; the result must not depend on the grid, and it must finish well
    # inside the bounded waits (no MOE_ERR_TIMEOUT)
    E, D, F, counts = 4, 1024, 512, [300, 40, 0, 129]
    n = sum(counts)
    g = torch.Generator().manual_seed(91)
    xp = torch.randn((n + 5, D), generator=g).to(torch.bfloat16)
    std = 1.0 / math.sqrt(D)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * std).to(torch.bfloat16)
    w2 = (torch.randn((E, D, F), generator=g) * std).to(torch.bfloat16)
    yp, off = run_ffn(xp, counts, w13, w2, F, max_ctas=ctas)
    ref = O.grouped_ffn(f64(xp)[:n], off, f64(w13), f64(w2))
    assert rel_err(f64(yp[:n]), ref) <= 1e-2
    full, _ = run_ffn(xp, counts, w13, w2, F)
    assert torch.equal(yp[:n], full[:n])    # the same bits on every grid


def test_grouped_ffn_all_experts_empty():
    # offsets all zero: no tile runs and the output rows stay untouched
    E, D, F, max_rows = 4, 128, 256, 64
    g = torch.Generator().manual_seed(5)
    xp = torch.randn((max_rows, D), generator=g).to(torch.bfloat16)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E, D, F), generator=g) * 0.05).to(torch.bfloat16)
    yp, _ = run_ffn(xp, [0] * E, w13, w2, F)
    assert torch.isnan(yp.float()).all()


@pytest.mark.parametrize("E,max_rows,variant", [(2, 128, 2), (2, 768, 3)])
def test_grouped_ffn_offsets_past_the_rows_run_nothing(E, max_rows, variant):
    # offsets implying more row blocks than the workspace's counters cover
    # (far past max_rows): both kernels report MOE_ERR_INVALID and run no
    # tile, so yp keeps its sentinels
    D, F = 128, 256
    assert L.moe_grouped_ffn_variant(E, D, F, max_rows,
                                     L.dtype_code(torch.bfloat16)) == variant
    g = torch.Generator().manual_seed(7)
    xp = torch.randn((max_rows, D), generator=g).to(torch.bfloat16).to(DEV)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * 0.05).to(
        torch.bfloat16).to(DEV)
    w2 = (torch.randn((E, D, F), generator=g) * 0.05).to(
        torch.bfloat16).to(DEV)
    off = torch.tensor([0, 3000, 6000][:E + 1], dtype=torch.int32, device=DEV)
    yp = torch.full((max_rows, D), float("nan"), dtype=torch.bfloat16,
                    device=DEV)
    ws = torch.empty(L.moe_grouped_ffn_workspace_size(
        E, D, F, max_rows, L.dtype_code(torch.bfloat16)), dtype=torch.uint8,
        device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_grouped_ffn(E, D, F, max_rows, L.dtype_code(torch.bfloat16), xp,
                      off, w13, w2, yp, ws, st)
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_INVALID
    assert torch.isnan(yp.float()).all()


def test_grouped_ffn_pairs_all_experts_empty():
    # the SM-pair kernel with every expert empty: the first claimed tile is
    # past the end, every pair leaves, the output rows stay untouched
    E, D, F, max_rows = 4, 128, 256, 1536
    assert L.moe_grouped_ffn_variant(E, D, F, max_rows,
                                     L.dtype_code(torch.bfloat16)) == 3
    g = torch.Generator().manual_seed(6)
    xp = torch.randn((max_rows, D), generator=g).to(torch.bfloat16)
    w13 = (torch.randn((E, 2 * F, D), generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn((E, D, F), generator=g) * 0.05).to(torch.bfloat16)
    yp, _ = run_ffn(xp, [0] * E, w13, w2, F)
    assert torch.isnan(yp.float()).all()


def test_row_movers_bound_rows():
    # a caller-supplied row id at or past max_rows is never read or written:
    # the pair is skipped, MOE_ERR_INDEX is raised, and canary rows past the
    # buffer's max_rows keep their contents
    T, k, D, rows, canary = 40, 2, 64, 100, 8
    dt = torch.bfloat16
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(rows, generator=g)[:T * k].clone()
    perm[5] = rows            # first row past the buffer
    perm[70] = rows + canary - 1   # the last canary row
    perm[9] = -1              # an ordinary drop
    dst = perm.to(torch.int32).to(DEV)
    ok = perm.clone()
    ok[ok >= rows] = -1       # what the movers must treat them as
    x = torch.randn((T, D), generator=g).to(dt)
    gate = torch.rand((T, k), generator=g).float()

    def fresh_status():
        return torch.zeros(1, dtype=torch.int32, device=DEV)

    buf = torch.full((rows + canary, D), float("nan"), dtype=dt, device=DEV)
    st = fresh_status()
    L.moe_permute(T, k, D, L.MOE_BF16, x.to(DEV), dst, buf, st,
                  max_rows=rows)
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_INDEX
    assert torch.isnan(buf[rows:].float()).all()
    for p in range(T * k):
        r = int(ok[p])
        if r >= 0:
            assert torch.equal(buf[r].cpu(), x[p // k])

    yp = torch.randn((rows + canary, D), generator=g).to(dt)
    y = torch.full((T, D), float("nan"), dtype=dt, device=DEV)
    st = fresh_status()
    L.moe_combine(T, k, D, L.MOE_BF16, yp.to(DEV), dst, gate.to(DEV), y, st,
                  max_rows=rows)
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_INDEX
    ref = O.combine(f64(yp), ok.numpy(), f64(gate), T, k)
    assert (np.abs(f64(y) - ref) <= np.abs(ref) * 2 ** -8 + 1e-6).all()

    dy = torch.randn((T, D), generator=g).to(dt).to(DEV)
    dyp = torch.full((rows + canary, D), float("nan"), dtype=dt, device=DEV)
    dgate = torch.full((T, k), float("nan"), device=DEV)
    st = fresh_status()
    L.moe_combine_backward(T, k, D, L.MOE_BF16, dy, yp.to(DEV), dst,
                           gate.to(DEV), dyp, dgate, st, max_rows=rows)
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_INDEX
    assert torch.isnan(dyp[rows:].float()).all()
    dg = dgate.cpu().numpy().reshape(-1)
    assert dg[5] == 0.0 and dg[70] == 0.0 and dg[9] == 0.0
    assert np.isfinite(dg).all()

    dx = torch.full((T, D), float("nan"), dtype=dt, device=DEV)
    st = fresh_status()
    L.moe_permute_backward(T, k, D, L.MOE_BF16, yp.to(DEV), dst, dx, st,
                           max_rows=rows)
    torch.cuda.synchronize()
    assert st.item() == L.MOE_ERR_INDEX
    ref = O.combine(f64(yp), ok.numpy(), np.ones((T, k)), T, k)
    assert (np.abs(f64(dx) - ref) <= np.abs(ref) * 2 ** -8 + 1e-6).all()

    # the same rows with the bad ids dropped raise nothing
    st = fresh_status()
    L.moe_permute(T, k, D, L.MOE_BF16, x.to(DEV), ok.to(torch.int32).to(DEV),
                  buf, st, max_rows=rows)
    torch.cuda.synchronize()
    assert st.item() == 0


def test_empty_batch_through_every_call():
    # T = 0 through route, permute and combine: each returns MOE_OK and
    # launches nothing (the C ABI raises on any other status)
    D, E, k = 256, 8, 2
    cfg = L.route_cfg(0, D, E, k, torch.bfloat16, "softmax_topk")
    x = torch.empty((0, D), dtype=torch.bfloat16, device=DEV)
    w = torch.randn((E, D), device=DEV).to(torch.bfloat16)
    ws = torch.empty(max(L.moe_route_workspace_size(cfg), 16),
                     dtype=torch.uint8, device=DEV)
    idx = torch.empty((0, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((0, k), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_route(cfg, x, w, None, None, idx, gate, None, ws, st)
    dst = torch.empty((0,), dtype=torch.int32, device=DEV)
    xp = torch.empty((0, D), dtype=torch.bfloat16, device=DEV)
    L.moe_permute(0, k, D, L.MOE_BF16, x, dst, xp)
    L.moe_combine(0, k, D, L.MOE_BF16, xp, dst, gate, x)
    torch.cuda.synchronize()
    assert st.item() == 0


# ------------------------------------------------------------ whole layer
def layer_from(wl, inp, keep_logits=True):
    return MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                    None if inp["w13"] is None else inp["w13"].to(DEV),
                    None if inp["w2"] is None else inp["w2"].to(DEV), F=wl.F,
                    score=wl.score,
                    sel_bias=None if inp["sel_bias"] is None
                    else inp["sel_bias"].to(DEV),
                    logit_offset=None if inp["logit_offset"] is None
                    else inp["logit_offset"].to(DEV),
                    capacity_factor=wl.capacity_factor, n_groups=wl.n_groups,
                    topk_groups=wl.topk_groups,
                    group_score_topk=wl.group_score_topk,
                    keep_logits=keep_logits)


def check_layer_vs_oracle(wl, inp, layer, y):
    logits = layer.logits.cpu().numpy()
    cap = O.expert_capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    assert layer.capacity == (cap or 0)
    ref = O.moe_forward(
        f64(inp["x"]), None, wl.k, wl.E, wl.R, wl.score,
        w13=None if inp["w13"] is None else f64(inp["w13"]),
        w2=None if inp["w2"] is None else f64(inp["w2"]),
        sel_bias=None if inp["sel_bias"] is None else inp["sel_bias"].numpy(),
        n_groups=wl.n_groups, topk_groups=wl.topk_groups,
        group_score_topk=wl.group_score_topk, capacity=cap, logits=logits)
    assert (i64(layer.topk_idx) == ref["topk_idx"]).all()
    assert np.abs(f64(layer.topk_gate) - ref["topk_gate"]).max() <= 2e-6
    assert i64(layer.expert_offsets).tolist() == ref["offsets"].tolist()
    assert i64(layer.dst_row).tolist() == ref["dst_row"].tolist()
    assert i64(layer.rank_send_counts).tolist() == \
        ref["rank_send_counts"].tolist()
    assert rel_err(f64(y), ref["y"]) <= tol_for(inp["x"].dtype)
    return ref


SMALL_LAYERS = [
    W.WORKLOADS["tiny_f32"],
    W.WORKLOADS["mixtral_bf16"].with_(T=256, D=512, F=1024),
    W.WORKLOADS["deepseek_bf16"].with_(T=192, D=1024, E=64, F=256),
    W.WORKLOADS["switch_bf16"].with_(T=2048, D=256, F=512),
    W.WORKLOADS["sweep_bf16_zipf_T4096"].with_(T=1000, D=1024),
]


@pytest.mark.parametrize("wl", SMALL_LAYERS, ids=lambda w: w.name)
def test_layer_parity_small(wl):
    inp = W.make_inputs(wl, device="cpu")
    layer = layer_from(wl, inp)
    x = inp["x"].to(DEV)
    if wl.routing is not None:
        # pre-drawn routing: run the router only for its logits check, then
        # feed the drawn ids and gates through layout/permute/combine
        y = layer.forward(x, inp["topk_idx"].to(DEV),
                          inp["topk_gate"].to(DEV))
        torch.cuda.synchronize()
        ref = O.moe_forward(f64(inp["x"]), None, wl.k, wl.E, wl.R, wl.score,
                            topk_idx=inp["topk_idx"].numpy(),
                            topk_gate=f64(inp["topk_gate"]))
        assert i64(layer.dst_row).tolist() == ref["dst_row"].tolist()
        assert rel_err(f64(y), ref["y"]) <= 1e-2
        assert rel_err(f64(y), f64(inp["x"])) <= 1e-2   # identity experts
        return
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref = check_layer_vs_oracle(wl, inp, layer, y)
    if wl.capacity_factor is not None:
        assert int(layer.n_dropped.item()) == ref["dropped"]


@pytest.mark.parametrize("wl", [
    W.WORKLOADS["mixtral_bf16"].with_(T=512, D=1024, F=1024),
    W.WORKLOADS["switch_bf16"].with_(T=2048, D=256, F=512),
    W.WORKLOADS["deepseek_bf16"].with_(T=256, D=1024, E=64, F=256)],
    ids=lambda w: w.name)
def test_forward_overlapped_matches_forward(wl):
    # micro-batches with the routing of batch i+1 on a second stream while
    # batch i's experts run on fewer CTAs: every batch's output equals the
    # plain forward pass of that batch, bit for bit (each batch keeps its own
    # routing decision and capacity)
    inp = W.make_inputs(wl, device="cpu")
    layer = layer_from(wl, inp)
    g = torch.Generator().manual_seed(77)
    xs = [(torch.randn((wl.T, wl.D), generator=g)).to(inp["x"].dtype).to(DEV)
          for _ in range(5)]
    ref = []
    for x in xs:
        ref.append(layer.forward(x).clone())
    ys = [torch.full_like(xs[0], float("nan")) for _ in xs]
    layer.forward_overlapped(xs, ys, ffn_ctas=64)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for a, b in zip(ys, ref):
        assert torch.equal(a, b)


def test_layer_repeatable_bitwise():
    wl = W.WORKLOADS["mixtral_bf16"].with_(T=300, D=256, F=512)
    inp = W.make_inputs(wl, device="cpu")
    layer = layer_from(wl, inp)
    x = inp["x"].to(DEV)
    y1 = layer.forward(x).clone()
    y2 = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
