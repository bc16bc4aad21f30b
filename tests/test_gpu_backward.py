"""GPU parity of the backward pass, through the C ABI, against the oracle's
float64 backward on the same seeded inputs.

Bars (each derived from the arithmetic, written into the checks):
  * aligned layout: bit-exact (integer work);
  * combine backward: dyp within one bf16 rounding of g*dy; dgate (an fp32
    dot product over D) within 1e-5 of sum_d |dy_d yp_d| + 1e-6;
  * router backward: dlogits within 1e-5 absolute (fp32 softmax/sigmoid
    algebra on gates <= 1); dw_r within 1e-4 of the matching sum of
    absolute terms (fp32 accumulation over T);
  * expert backward (bf16 tensor-core GEMMs with dH, [dG|dU] and H rounded
    to bf16 between them, as in the forward's H): max|got - ref| /
    max|ref| <= 2e-2 per gradient.  Each of the two bf16 roundings on the
    way adds at most 2^-9 relative per element; the bound leaves room for
    their accumulation over the contraction;
  * whole layer (forward_train + backward): the same 2e-2 bar on dx, dw_r,
    dw13, dw2, and the forward output within the forward's 1e-2 bar.
"""
import math

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from combine_router_gemm_top_b300 import _lib as L
from combine_router_gemm_top_b300 import workloads as W
from combine_router_gemm_top_b300.layer import MoELayer

pytestmark = pytest.mark.gpu

DEV = "cuda"
I32 = dict(dtype=torch.int32, device=DEV)
BF = torch.bfloat16


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def i64(t):
    return t.detach().to("cpu", torch.int64).numpy()


def rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return np.abs(got - ref).max() / (den if den > 0 else 1.0)


def routing(T, k, E, seed, skew=0.0):
    g = torch.Generator().manual_seed(seed)
    logw = -skew * torch.log(torch.arange(1, E + 1, dtype=torch.float64))
    u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_min(1e-300)
    return torch.topk(logw - torch.log(-torch.log(u)), k, dim=1).indices.to(
        torch.int32)


def layout_on_gpu(idx, E, cap=0):
    T, k = idx.shape
    P = T * k
    ws = torch.empty(L.moe_dispatch_layout_workspace_size(T, k, E),
                     dtype=torch.uint8, device=DEV)
    o = dict(counts=torch.empty(E, **I32), off=torch.empty(E + 1, **I32),
             dst=torch.empty(P, **I32), src=torch.empty(P, **I32),
             nk=torch.empty(1, **I32), nd=torch.empty(1, **I32),
             rc=torch.empty(1, **I32), rd=torch.empty(1, **I32))
    st = torch.zeros(1, **I32)
    L.moe_dispatch_layout(T, k, E, 1, cap, idx.to(DEV), o["counts"], o["off"],
                          o["dst"], o["src"], o["nk"], o["nd"], o["rc"],
                          o["rd"], ws, st)
    return o, st


# ------------------------------------------------------ aligned layout -----
@pytest.mark.parametrize("T,k,E,cap,align", [(300, 2, 7, 90, 64),
                                             (1000, 8, 64, 0, 64),
                                             (5, 1, 3, 0, 16),
                                             (2048, 2, 8, 0, 128)])
def test_aligned_layout_bit_exact(T, k, E, cap, align):
    idx = routing(T, k, E, seed=T + E, skew=1.0)
    o, st = layout_on_gpu(idx, E, cap)
    dst_a = torch.full((T * k,), -9, **I32)
    off_a = torch.full((E + 1,), -9, **I32)
    L.moe_aligned_layout(T, k, E, align, idx.to(DEV), o["dst"], o["off"],
                         dst_a, off_a, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    lay = O.dispatch_layout(idx.numpy(), E, 1, cap or None)
    ref = O.aligned_layout(lay, E, align)
    assert i64(off_a).tolist() == ref["offsets_aligned"].tolist()
    assert i64(dst_a).tolist() == ref["dst_row_aligned"].tolist()


# ------------------------------------------------------ combine backward ---
@pytest.mark.parametrize("T,k,E,D,cap,dt", [(257, 2, 8, 512, 70, BF),
                                            (100, 8, 32, 1024, 0, BF),
                                            (64, 1, 4, 64, 0, torch.float32)])
def test_combine_backward_parity(T, k, E, D, cap, dt):
    idx = routing(T, k, E, seed=D + k)
    o, st = layout_on_gpu(idx, E, cap)
    rows = T * k
    g = torch.Generator().manual_seed(T)
    yp = torch.randn((rows, D), generator=g).to(dt)
    dy = torch.randn((T, D), generator=g).to(dt)
    gate = torch.rand((T, k), generator=g)
    dyp = torch.full((rows, D), float("nan"), dtype=dt, device=DEV)
    dgate = torch.full((T, k), float("nan"), device=DEV)
    L.moe_combine_backward(T, k, D, L.dtype_code(dt), dy.to(DEV), yp.to(DEV),
                           o["dst"], gate.to(DEV), dyp, dgate)
    torch.cuda.synchronize()
    dst = i64(o["dst"])
    ydy, yyp, yg = f64(dy), f64(yp), gate.double().numpy()
    got, gd = f64(dyp), f64(dgate)
    ulp = 2.0 ** -8 if dt == BF else 2.0 ** -23
    for t in range(T):
        for j in range(k):
            r = dst[t * k + j]
            if r < 0:
                assert gd[t, j] == 0.0
                continue
            ref = yg[t, j] * ydy[t]
            assert (np.abs(got[r] - ref) <= ulp * np.abs(ref) + 1e-30).all()
            dot = ydy[t] @ yyp[r]
            bound = 1e-5 * np.abs(ydy[t] * yyp[r]).sum() + 1e-6
            assert abs(gd[t, j] - dot) <= bound


# ------------------------------------------------------ expert backward ----
def aligned_inputs(counts, D, F, seed, align=64):
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)])
    off_a = np.concatenate([[0], np.cumsum([(c + align - 1) // align * align
                                            for c in counts])])
    rows = int(off_a[-1]) + align
    g = torch.Generator().manual_seed(seed)
    std = 1.0 / math.sqrt(D)
    xp = torch.zeros((rows, D))
    dyp = torch.zeros((rows, D))
    for e in range(E):
        c = counts[e]
        xp[off_a[e]:off_a[e] + c] = torch.randn((c, D), generator=g)
        dyp[off_a[e]:off_a[e] + c] = torch.randn((c, D), generator=g)
    w13 = torch.randn((E, 2 * F, D), generator=g) * std
    w2 = torch.randn((E, D, F), generator=g) / math.sqrt(F)
    return (xp.to(BF), dyp.to(BF), w13.to(BF), w2.to(BF),
            off_a.astype(np.int32), rows)


def run_ffn_backward(xp, dyp, w13, w2, off_a, rows):
    E, twoF, D = w13.shape
    F = twoF // 2
    ws = torch.empty(L.moe_grouped_ffn_backward_workspace_size(
        E, D, F, rows, L.MOE_BF16), dtype=torch.uint8, device=DEV)
    dxp = torch.full((rows, D), float("nan"), dtype=BF, device=DEV)
    dw13 = torch.full((E, 2 * F, D), float("nan"), device=DEV)
    dw2 = torch.full((E, D, F), float("nan"), device=DEV)
    st = torch.zeros(1, **I32)
    L.moe_grouped_ffn_backward(E, D, F, rows, L.MOE_BF16, xp.to(DEV),
                               dyp.to(DEV), torch.tensor(off_a, device=DEV),
                               w13.to(DEV), w2.to(DEV), dxp, dw13, dw2, ws,
                               st)
    torch.cuda.synchronize()
    return dxp, dw13, dw2, int(st.item())


FFN_BWD_CASES = [
    # counts per expert, D, F
    ([64, 128, 0, 37], 128, 128),
    ([200, 1, 300], 256, 256),
    ([512, 448], 512, 384),
    ([130, 0, 0, 77, 64, 5, 256, 190], 256, 128),
]


@pytest.mark.parametrize("case", FFN_BWD_CASES)
def test_grouped_ffn_backward_parity(case):
    counts, D, F = case
    E = len(counts)
    xp, dyp, w13, w2, off_a, rows = aligned_inputs(counts, D, F,
                                                   seed=D + F + E)
    dxp, dw13, dw2, st = run_ffn_backward(xp, dyp, w13, w2, off_a, rows)
    assert st == 0
    X, DY, W13, W2 = f64(xp), f64(dyp), f64(w13), f64(w2)
    ref_dxp = np.zeros_like(X)
    for e in range(E):
        a, c = int(off_a[e]), counts[e]
        w1, w3 = O.split_w13(W13[e])
        if c == 0:
            assert (dw13[e] == 0).all() and (dw2[e] == 0).all()
            continue
        dh, dw1, dw3, dw2e = O.expert_backward(X[a:a + c], w1, w3, W2[e],
                                               DY[a:a + c])
        ref_dxp[a:a + c] = dh
        assert rel(f64(dw13[e, :F]), dw1) <= 2e-2
        assert rel(f64(dw13[e, F:]), dw3) <= 2e-2
        assert rel(f64(dw2[e]), dw2e) <= 2e-2
    n_rows = int(off_a[E])                # rows past the layout: unwritten
    got = f64(dxp)[:n_rows]
    assert np.isfinite(got).all()
    assert rel(got, ref_dxp[:n_rows]) <= 2e-2
    assert torch.isnan(dxp[n_rows:].float()).all()
    # padding rows of the aligned layout stay zero
    for e in range(E):
        a, c, b = int(off_a[e]), counts[e], int(off_a[e + 1])
        assert (got[a + c:b] == 0).all()


def test_grouped_ffn_backward_rejects_unaligned_offsets():
    counts, D, F = [64, 64], 128, 128
    xp, dyp, w13, w2, off_a, rows = aligned_inputs(counts, D, F, seed=1)
    bad = off_a.copy()
    bad[1] = 60
    _, dw13, _, st = run_ffn_backward(xp, dyp, w13, w2, bad, rows)
    assert st == L.MOE_ERR_INVALID
    assert torch.isnan(dw13).all()          # no weight gradient written


# ------------------------------------------------------ router backward ----
@pytest.mark.parametrize("T,D,E,k,score,groups", [
    (300, 256, 8, 2, "softmax_topk", (1, 1, 0)),
    (513, 128, 64, 1, "softmax_full", (1, 1, 0)),
    (257, 512, 256, 8, "sigmoid_bias", (8, 4, 2)),
    (64, 64, 16, 4, "sigmoid_bias", (1, 1, 0)),
    # tensor-core path: D not a multiple of 256, E = 3 x 64, split-K dW_r
    (200, 384, 128, 8, "softmax_topk", (1, 1, 0)),
    (130, 1024, 192, 6, "softmax_topk", (1, 1, 0)),
    (1000, 512, 64, 2, "sigmoid_bias", (4, 2, 2)),
    (1, 64, 64, 1, "softmax_topk", (1, 1, 0))])
def test_route_backward_parity(T, D, E, k, score, groups):
    g = torch.Generator().manual_seed(T + E)
    x = torch.randn((T, D), generator=g).to(BF)
    w_r = (torch.randn((E, D), generator=g) / math.sqrt(D)).to(BF)
    logits = torch.randn((T, E), generator=g) * 2.0
    idx, _ = O.route_from_logits(logits.numpy(), k, score, None, *groups)
    dgate = torch.randn((T, k), generator=g)
    dx0 = torch.randn((T, D), generator=g).to(BF)
    cfg = L.route_cfg(T, D, E, k, BF, score, *groups)
    dl = torch.full((T, E), float("nan"), device=DEV)
    dwr = torch.full((E, D), float("nan"), device=DEV)
    dx = dx0.to(DEV)
    st = torch.zeros(1, **I32)
    ws = torch.empty(L.moe_route_backward_workspace_size(cfg),
                     dtype=torch.uint8, device=DEV)
    L.moe_route_backward(cfg, x.to(DEV), w_r.to(DEV), logits.to(DEV),
                         torch.tensor(idx, device=DEV), dgate.to(DEV), dl,
                         dwr, dx, ws, st)
    torch.cuda.synchronize()
    ref_dl = np.stack([O.gate_backward(logits[t].numpy(), idx[t],
                                       dgate[t].numpy(), score)
                       for t in range(T)])
    assert np.abs(f64(dl) - ref_dl).max() <= 1e-5
    X, WR = f64(x), f64(w_r)
    ref_dwr = ref_dl.T @ X
    bound = 1e-4 * (np.abs(ref_dl).T @ np.abs(X)) + 1e-6
    assert (np.abs(f64(dwr) - ref_dwr) <= bound).all()
    ref_dx = f64(dx0) + ref_dl @ WR
    assert rel(f64(dx), ref_dx) <= 1e-2


# ------------------------------------------------------ whole layer --------
BWD_LAYERS = [
    W.WORKLOADS["mixtral_bf16"].with_(T=256, D=512, F=1024),
    W.WORKLOADS["deepseek_bf16"].with_(T=192, D=1024, E=64, F=256),
    W.WORKLOADS["switch_bf16"].with_(T=1024, D=256, F=512),
]


@pytest.mark.parametrize("wl", BWD_LAYERS, ids=lambda w: w.name)
def test_layer_backward_matches_oracle(wl):
    inp = W.make_inputs(wl, device="cpu")
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), F=wl.F,
                     score=wl.score,
                     sel_bias=None if inp["sel_bias"] is None
                     else inp["sel_bias"].to(DEV),
                     logit_offset=None if inp["logit_offset"] is None
                     else inp["logit_offset"].to(DEV),
                     capacity_factor=wl.capacity_factor, n_groups=wl.n_groups,
                     topk_groups=wl.topk_groups,
                     group_score_topk=wl.group_score_topk, keep_logits=True)
    x = inp["x"].to(DEV)
    y = layer.forward_train(x).clone()
    g = torch.Generator().manual_seed(wl.T)
    dy = torch.randn((wl.T, wl.D), generator=g).to(BF)
    dx, dw_r, dw13, dw2 = layer.backward(dy.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    cap = O.expert_capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    ref = O.moe_backward(
        f64(inp["x"]), f64(inp["w_r"]), f64(dy), wl.k, wl.E, wl.R, wl.score,
        w13=f64(inp["w13"]), w2=f64(inp["w2"]),
        sel_bias=None if inp["sel_bias"] is None else inp["sel_bias"].numpy(),
        n_groups=wl.n_groups, topk_groups=wl.topk_groups,
        group_score_topk=wl.group_score_topk, capacity=cap,
        logits=layer.logits.cpu().numpy())
    fw = ref["forward"]
    assert (i64(layer.topk_idx) == fw["topk_idx"]).all()
    assert rel(f64(y), fw["y"]) <= 1e-2
    for got, want in ((dx, ref["dx"]), (dw_r, ref["dw_r"]),
                      (dw13, ref["dw13"]), (dw2, ref["dw2"])):
        assert np.isfinite(f64(got)).all()
        assert rel(f64(got), want) <= 2e-2


# ------------------------------------------------------ fp32 backward ------
@pytest.mark.parametrize("counts,D,F", [([10, 0, 37, 64, 1], 64, 96),
                                        ([130, 70, 5], 40, 128)])
def test_grouped_ffn_backward_fp32_parity(counts, D, F):
    # the fp32 path takes any offsets and any D, F; fp32 accumulation over
    # K <= 256 terms keeps it within 1e-5 of the float64 oracle
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off[-1]) + 3
    g = torch.Generator().manual_seed(D + F)
    xp = torch.randn((rows, D), generator=g)
    dyp = torch.randn((rows, D), generator=g)
    w13 = torch.randn((E, 2 * F, D), generator=g) / math.sqrt(D)
    w2 = torch.randn((E, D, F), generator=g) / math.sqrt(F)
    ws = torch.empty(L.moe_grouped_ffn_backward_workspace_size(
        E, D, F, rows, L.MOE_F32), dtype=torch.uint8, device=DEV)
    dxp = torch.full((rows, D), float("nan"), device=DEV)
    dw13 = torch.full((E, 2 * F, D), float("nan"), device=DEV)
    dw2 = torch.full((E, D, F), float("nan"), device=DEV)
    st = torch.zeros(1, **I32)
    L.moe_grouped_ffn_backward(E, D, F, rows, L.MOE_F32, xp.to(DEV),
                               dyp.to(DEV), torch.tensor(off, device=DEV),
                               w13.to(DEV), w2.to(DEV), dxp, dw13, dw2, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    X, DY, W13, W2 = f64(xp), f64(dyp), f64(w13), f64(w2)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b == a:
            assert (dw13[e] == 0).all() and (dw2[e] == 0).all()
            continue
        w1, w3 = O.split_w13(W13[e])
        dh, dw1, dw3, dw2e = O.expert_backward(X[a:b], w1, w3, W2[e],
                                               DY[a:b])
        assert rel(f64(dxp[a:b]), dh) <= 1e-5
        assert rel(f64(dw13[e, :F]), dw1) <= 1e-5
        assert rel(f64(dw13[e, F:]), dw3) <= 1e-5
        assert rel(f64(dw2[e]), dw2e) <= 1e-5


@pytest.mark.parametrize("wl", [
    W.WORKLOADS["tiny_f32"],
    W.WORKLOADS["deepseek_bf16"].with_(name="deepseek_f32_small", T=96, D=64,
                                       E=32, F=48, dtype="f32"),
    W.WORKLOADS["switch_bf16"].with_(name="switch_f32_small", T=512, D=32,
                                     E=16, F=64, dtype="f32"),
], ids=lambda w: w.name)
def test_layer_backward_fp32_tight(wl):
    # the whole fp32 training step against the float64 oracle at the fp32
    # bar: combine, expert, permute and router backward all in fp32
    inp = W.make_inputs(wl, device="cpu")
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), F=wl.F,
                     score=wl.score,
                     sel_bias=None if inp["sel_bias"] is None
                     else inp["sel_bias"].to(DEV),
                     logit_offset=None if inp["logit_offset"] is None
                     else inp["logit_offset"].to(DEV),
                     capacity_factor=wl.capacity_factor, n_groups=wl.n_groups,
                     topk_groups=wl.topk_groups,
                     group_score_topk=wl.group_score_topk, keep_logits=True)
    x = inp["x"].to(DEV)
    y = layer.forward_train(x).clone()
    g = torch.Generator().manual_seed(wl.T + 1)
    dy = torch.randn((wl.T, wl.D), generator=g)
    dx, dw_r, dw13, dw2 = layer.backward(dy.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    cap = O.expert_capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    ref = O.moe_backward(
        f64(inp["x"]), f64(inp["w_r"]), f64(dy), wl.k, wl.E, wl.R, wl.score,
        w13=f64(inp["w13"]), w2=f64(inp["w2"]),
        sel_bias=None if inp["sel_bias"] is None else inp["sel_bias"].numpy(),
        logit_offset=None if inp["logit_offset"] is None
        else inp["logit_offset"].numpy(),
        n_groups=wl.n_groups, topk_groups=wl.topk_groups,
        group_score_topk=wl.group_score_topk, capacity=cap,
        logits=layer.logits.cpu().numpy())
    assert (i64(layer.topk_idx) == ref["forward"]["topk_idx"]).all()
    assert rel(f64(y), ref["forward"]["y"]) <= 1e-5
    for got, want in ((dx, ref["dx"]), (dw_r, ref["dw_r"]),
                      (dw13, ref["dw13"]), (dw2, ref["dw2"])):
        assert rel(f64(got), want) <= 1e-5
