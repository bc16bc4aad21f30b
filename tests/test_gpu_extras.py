"""GPU parity of the calls beyond the five-step path, through the C ABI,
against the CPU oracle on the same seeded inputs:

  * moe_router_stats: routed counts bit-exact; f within one fp32 rounding
    of the exact ratio; P within 1e-6 absolute (fp32 probabilities summed in
    fp64, P <= 1); L_aux within 1e-5 relative;
  * moe_router_bias_update: bit-exact (one fp32 add per expert);
  * moe_dispatch_matrix, moe_padded_layout, moe_pad_fill: bit-exact
    (integer work and copies);
  * the layer on the padded static-capacity layout: the same bars as the
    compact layer (integers bit-exact, output within 1e-2 relative in bf16);
  * node-limited routing (groups = destination ranks): ids bit-exact and
    every token reaches at most the allowed number of ranks.
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


def i64(t):
    return t.detach().to("cpu", torch.int64).numpy()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rand_routing(T, k, E, seed, skew=0.0):
    """k distinct experts per token (Gumbel top-k over log-weights)."""
    g = torch.Generator().manual_seed(seed)
    logw = -skew * torch.log(torch.arange(1, E + 1, dtype=torch.float64))
    u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_min(1e-300)
    keys = logw - torch.log(-torch.log(u))
    return torch.topk(keys, k, dim=1).indices.to(torch.int32)


# ------------------------------------------------------- router statistics
def run_stats(logits, idx, E, score, alpha):
    T, k = idx.shape
    ws = torch.empty(max(L.moe_router_stats_workspace_size(T, E), 16),
                     dtype=torch.uint8, device=DEV)
    f = torch.full((E,), float("nan"), device=DEV)
    P = torch.full((E,), float("nan"), device=DEV)
    cnt = torch.full((E,), -1, **I32)
    loss = torch.full((1,), float("nan"), device=DEV)
    st = torch.zeros(1, **I32)
    L.moe_router_stats(T, E, k, score, logits.to(DEV), idx.to(DEV), alpha, f,
                       P, cnt, loss, ws, st)
    torch.cuda.synchronize()
    return f64(f), f64(P), i64(cnt), float(loss.item()), int(st.item())


STATS_CASES = [
    # T, E, k, score, logit scale, skew
    (1, 8, 2, "softmax_topk", 1.0, 0.0),
    (37, 8, 2, "softmax_topk", 3.0, 0.0),
    (1000, 64, 1, "softmax_full", 2.0, 1.2),
    (4096, 256, 8, "sigmoid_bias", 1.0, 0.0),
    (2049, 128, 8, "softmax_topk", 0.5, 1.2),
    (300, 40, 3, "sigmoid_bias", 4.0, 0.5),
]


@pytest.mark.parametrize("case", STATS_CASES)
def test_router_stats_parity(case):
    T, E, k, score, scale, skew = case
    g = torch.Generator().manual_seed(T + E)
    logits = (torch.randn((T, E), generator=g) * scale).float()
    idx = rand_routing(T, k, E, seed=T * 3 + k, skew=skew)
    f, P, cnt, loss, st = run_stats(logits, idx, E, score, alpha=0.01)
    assert st == 0
    ref = O.router_stats(logits.numpy(), idx.numpy(), E, score, 0.01)
    assert cnt.tolist() == ref["counts_routed"].tolist()
    assert np.abs(f - ref["f"]).max() <= 2.0 ** -24 * np.abs(ref["f"]).max()
    assert np.abs(P - ref["P"]).max() <= 1e-6
    assert abs(loss - ref["aux_loss"]) <= 1e-5 * abs(ref["aux_loss"])


def test_router_stats_balanced_closed_form():
    # equal logits and perfectly even routing: L_aux = alpha exactly up to
    # rounding
    T, E, k = 512, 16, 4
    idx = torch.tensor([[(t * k + j) % E for j in range(k)]
                        for t in range(T)], dtype=torch.int32)
    f, P, cnt, loss, st = run_stats(torch.zeros((T, E)), idx, E,
                                    "softmax_topk", alpha=0.02)
    assert st == 0 and (cnt == T * k // E).all()
    assert abs(loss - 0.02) <= 1e-7


def test_router_stats_reports_bad_ids():
    T, E, k = 64, 8, 2
    idx = rand_routing(T, k, E, seed=1)
    idx[5, 1] = E + 3
    f, P, cnt, loss, st = run_stats(torch.zeros((T, E)), idx, E,
                                    "softmax_topk", alpha=1.0)
    assert st == L.MOE_ERR_INDEX
    assert cnt.sum() == T * k - 1


def test_router_stats_repeatable_bitwise():
    T, E, k = 3000, 64, 4
    g = torch.Generator().manual_seed(9)
    logits = torch.randn((T, E), generator=g)
    idx = rand_routing(T, k, E, seed=2)
    a = run_stats(logits, idx, E, "softmax_topk", 0.1)
    b = run_stats(logits, idx, E, "softmax_topk", 0.1)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all() and a[3] == b[3]


@pytest.mark.parametrize("E,T,k", [(8, 100, 2), (256, 4096, 8), (3, 5, 1)])
def test_bias_update_bit_exact(E, T, k):
    idx = rand_routing(T, k, E, seed=E, skew=1.0)
    cnt = torch.bincount(idx.reshape(-1).long(), minlength=E).to(torch.int32)
    g = torch.Generator().manual_seed(E)
    bias = (torch.rand(E, generator=g) * 0.2 - 0.1).float()
    d_bias = bias.to(DEV)
    L.moe_router_bias_update(T, k, E, cnt.to(DEV), 0.001, d_bias)
    torch.cuda.synchronize()
    ref = O.bias_update(bias.numpy(), cnt.numpy(), T, k, 0.001)
    assert (d_bias.cpu().numpy() == ref).all()


# --------------------------------------------------------- dispatch matrix
def run_matrix(idx, E, n_src, n_dst, dst_row=None):
    T, k = idx.shape
    m = torch.full((n_src * n_dst,), -5, **I32)
    st = torch.zeros(1, **I32)
    L.moe_dispatch_matrix(T, k, E, n_src, n_dst, idx.to(DEV),
                          None if dst_row is None else dst_row.to(DEV), m, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return i64(m).reshape(n_src, n_dst)


MATRIX_CASES = [
    # T, k, E, n_src, n_dst, skew
    (8 * 1024, 2, 64, 8, 8, 0.0),     # the pages' simulation shape
    (4, 2, 4, 2, 2, 0.0),
    (65536, 8, 128, 8, 8, 1.2),
    (3000, 1, 64, 3, 16, 1.0),
    (4096, 8, 256, 16, 8, 0.0),
]


@pytest.mark.parametrize("case", MATRIX_CASES)
def test_dispatch_matrix_bit_exact(case):
    T, k, E, n_src, n_dst, skew = case
    idx = rand_routing(T, k, E, seed=T + E, skew=skew)
    m = run_matrix(idx, E, n_src, n_dst)
    ref = O.dispatch_matrix(idx.numpy(), n_src, n_dst, E)
    assert (m == ref).all()
    assert (m.sum(axis=1) == T // n_src * k).all()


def test_dispatch_matrix_counts_kept_pairs_only():
    T, k, E, R = 2048, 2, 16, 4
    idx = rand_routing(T, k, E, seed=4, skew=1.5)
    cap = 200
    lay = O.dispatch_layout(idx.numpy(), E, R, cap)
    assert lay["dropped"] > 0
    dst = torch.tensor(lay["dst_row"], dtype=torch.int32)
    m = run_matrix(idx, E, 4, R, dst)
    ref = O.dispatch_matrix(idx.numpy(), 4, R, E, lay["dst_row"])
    assert (m == ref).all()
    assert (m.sum(axis=0) == lay["rank_send_counts"]).all()


def test_dispatch_matrix_page_worked_example():
    idx = torch.tensor([[0, 2], [1, 3], [0, 1], [2, 3]], dtype=torch.int32)
    assert run_matrix(idx, 4, 2, 2).tolist() == [[2, 2], [2, 2]]
    assert run_matrix(idx, 4, 4, 2).tolist() == [[1, 1], [1, 1], [2, 0],
                                                  [0, 2]]


# ------------------------------------------------------ padded layout -----
def padded_from_layer(layer, cap):
    T, k, E, D = layer.T, layer.k, layer.E, layer.D
    P = T * k
    dst_p = torch.full((P,), -9, **I32)
    off_p = torch.full((E + 1,), -9, **I32)
    st = torch.zeros(1, **I32)
    L.moe_padded_layout(T, k, E, cap, layer.topk_idx, layer.dst_row,
                        layer.expert_offsets, dst_p, off_p, st)
    xpad = torch.full((E * cap, D), float("nan"), dtype=layer.dtype,
                      device=DEV)
    L.moe_pad_fill(E, cap, D, layer.dcode, layer.expert_counts, xpad)
    return dst_p, off_p, xpad, st


@pytest.mark.parametrize("wl", [
    W.WORKLOADS["tiny_f32"],
    W.WORKLOADS["switch_bf16"].with_(T=2048, D=256, F=512),
    W.WORKLOADS["mixtral_bf16"].with_(T=512, D=512, F=1024,
                                      capacity_factor=1.0),
], ids=lambda w: w.name)
def test_padded_layer_matches_oracle(wl):
    inp = W.make_inputs(wl, device="cpu")
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), F=wl.F,
                     score=wl.score,
                     logit_offset=None if inp["logit_offset"] is None
                     else inp["logit_offset"].to(DEV),
                     capacity_factor=wl.capacity_factor, keep_logits=True)
    cap = layer.capacity
    assert cap > 0
    x = inp["x"].to(DEV)
    layer.route(x)
    layer.dispatch_layout()
    dst_p, off_p, xpad, st = padded_from_layer(layer, cap)
    L.moe_permute(wl.T, wl.k, wl.D, layer.dcode, x, dst_p, xpad)
    ypad = torch.full_like(xpad, float("nan"))
    ws = torch.empty(L.moe_grouped_ffn_workspace_size(
        wl.E, wl.D, wl.F, wl.E * cap, layer.dcode), dtype=torch.uint8,
        device=DEV)
    L.moe_grouped_ffn(wl.E, wl.D, wl.F, wl.E * cap, layer.dcode, xpad, off_p,
                      layer.w13, layer.w2, ypad, ws, st)
    y = torch.empty_like(x)
    L.moe_combine(wl.T, wl.k, wl.D, layer.dcode, ypad, dst_p,
                  layer.topk_gate, y)
    torch.cuda.synchronize()
    assert st.item() == 0 and layer.device_status() == 0

    lay = O.dispatch_layout(i64(layer.topk_idx), wl.E, wl.R, cap)
    pad = O.padded_layout(lay, wl.E, cap)
    assert i64(dst_p).tolist() == pad["dst_row_padded"].tolist()
    assert i64(off_p).tolist() == pad["offsets_padded"].tolist()
    xref = O.permute_padded(f64(x), pad["src_pair_padded"], wl.k)
    assert (f64(xpad) == xref).all()             # copies and exact zeros
    ref = O.moe_forward(f64(inp["x"]), None, wl.k, wl.E, wl.R, wl.score,
                        w13=f64(inp["w13"]), w2=f64(inp["w2"]),
                        capacity=cap, logits=layer.logits.cpu().numpy())
    tol = 1e-5 if wl.dtype == "f32" else 1e-2
    err = np.abs(f64(y) - ref["y"]).max() / np.abs(ref["y"]).max()
    assert err <= tol
    # padding rows of the static-shape FFN output are exactly zero
    pad_rows = torch.tensor(pad["src_pair_padded"] < 0, device=DEV)
    assert (ypad[pad_rows] == 0).all()


def test_pad_fill_leaves_kept_rows():
    E, cap, D = 5, 7, 64
    counts = torch.tensor([0, 7, 3, 1, 6], dtype=torch.int32)
    buf = torch.full((E * cap, D), 3.0, dtype=torch.bfloat16, device=DEV)
    L.moe_pad_fill(E, cap, D, L.MOE_BF16, counts.to(DEV), buf)
    torch.cuda.synchronize()
    b = buf.float().cpu()
    for e in range(E):
        c = int(counts[e])
        assert (b[e * cap:e * cap + c] == 3.0).all()
        assert (b[e * cap + c:(e + 1) * cap] == 0.0).all()


# ------------------------------------------------- node-limited routing ---
@pytest.mark.parametrize("R,M", [(8, 4), (8, 2), (16, 3)])
def test_node_limited_routing(R, M):
    # groups = destination ranks: each token picks its M best ranks (by the
    # sum of its top k/M scores there) before the top-k
    T, D, E, k = 1024, 512, 128, 8
    g = torch.Generator().manual_seed(R * 10 + M)
    x = torch.randn((T, D), generator=g).to(torch.bfloat16)
    w = (torch.randn((E, D), generator=g) / math.sqrt(D)).to(torch.bfloat16)
    bias = ((torch.rand(E, generator=g) * 2 - 1) * 0.1).float()
    per = max(1, k // M)
    cfg = L.route_cfg(T, D, E, k, torch.bfloat16, "sigmoid_bias", R, M, per)
    ws = torch.empty(L.moe_route_workspace_size(cfg), dtype=torch.uint8,
                     device=DEV)
    idx = torch.empty((T, k), **I32)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, **I32)
    L.moe_route(cfg, x.to(DEV), w.to(DEV), None, bias.to(DEV), idx, gate,
                logits, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ridx, _ = O.route_from_logits(logits.cpu().numpy(), k, "sigmoid_bias",
                                  bias.numpy(), R, M, per)
    got = i64(idx)
    assert (got == ridx).all()
    ranks = got // (E // R)
    assert max(len(set(r.tolist())) for r in ranks) <= M
    m = run_matrix(idx.cpu(), E, 4, R)
    assert m.sum() == T * k


def test_padded_layer_mode_equals_compact_on_kept_pairs():
    # MoELayer(padded=True) runs the static-capacity layout: the same kept
    # pairs as the compact layer, and both outputs within the bf16 bound of
    # the oracle
    wl = W.WORKLOADS["switch_bf16"].with_(T=1024, D=256, F=256)
    inp = W.make_inputs(wl, device="cpu")
    kw = dict(F=wl.F, score=wl.score,
              logit_offset=inp["logit_offset"].to(DEV),
              capacity_factor=wl.capacity_factor, keep_logits=True)
    a = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                 inp["w13"].to(DEV), inp["w2"].to(DEV), **kw)
    b = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                 inp["w13"].to(DEV), inp["w2"].to(DEV), padded=True, **kw)
    x = inp["x"].to(DEV)
    ya = a.forward(x).clone()
    yb = b.forward(x).clone()
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
    assert (i64(a.dst_row) == i64(b.dst_row)).all()
    ref = O.moe_forward(f64(inp["x"]), None, wl.k, wl.E, wl.R, wl.score,
                        w13=f64(inp["w13"]), w2=f64(inp["w2"]),
                        capacity=a.capacity, logits=a.logits.cpu().numpy())
    for y in (ya, yb):
        err = np.abs(f64(y) - ref["y"]).max() / np.abs(ref["y"]).max()
        assert err <= 1e-2


def test_host_stream_matches_forward_bitwise():
    # forward_host_stream overlaps each batch's copies with its neighbours'
    # compute; every batch's output must equal forward() on that batch
    wl = W.WORKLOADS["mixtral_bf16"].with_(T=256, D=512, F=1024)
    inp = W.make_inputs(wl, device="cpu")
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), F=wl.F,
                     score=wl.score)
    g = torch.Generator().manual_seed(3)
    xs = [torch.randn((wl.T, wl.D), generator=g).to(torch.bfloat16)
          .pin_memory() for _ in range(5)]
    ys = [torch.full((wl.T, wl.D), float("nan"),
                     dtype=torch.bfloat16).pin_memory() for _ in range(5)]
    layer.forward_host_stream(xs, ys)
    torch.cuda.synchronize()
    for xh, yh in zip(xs, ys):
        ref = layer.forward(xh.to(DEV)).cpu()
        torch.cuda.synchronize()
        assert torch.equal(yh, ref)
    # the single-batch form: copy in, run, copy out on one stream
    x_dev = torch.empty((wl.T, wl.D), dtype=torch.bfloat16, device=DEV)
    y1 = torch.full((wl.T, wl.D), float("nan"), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xs[2], y1, x_dev)
    torch.cuda.synchronize()
    assert torch.equal(y1, ys[2])
    assert layer.device_status() == 0


@pytest.mark.parametrize("wl", [
    W.WORKLOADS["tiny_f32"],
    W.WORKLOADS["mixtral_bf16"].with_(T=256, D=512, F=1024),
    W.WORKLOADS["deepseek_bf16"].with_(T=192, D=1024, E=64, F=256),
], ids=lambda w: w.name)
def test_graph_replay_matches_eager_bitwise(wl):
    # the captured pass replays on new data in the same input buffer and
    # gives exactly what the eager pass gives
    inp = W.make_inputs(wl, device="cpu")
    kw = dict(F=wl.F, score=wl.score,
              sel_bias=None if inp["sel_bias"] is None
              else inp["sel_bias"].to(DEV),
              capacity_factor=wl.capacity_factor, n_groups=wl.n_groups,
              topk_groups=wl.topk_groups,
              group_score_topk=wl.group_score_topk)
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), **kw)
    x = inp["x"].to(DEV)
    replay = layer.capture(x)
    g = torch.Generator().manual_seed(5)
    for _ in range(3):
        new = torch.randn(x.shape, generator=g).to(x.dtype)
        x.copy_(new.to(DEV))
        y_graph = replay().clone()
        y_eager = layer.forward(new.to(DEV)).clone()
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y_eager)
    assert layer.device_status() == 0


def test_graph_replay_of_training_step():
    wl = W.WORKLOADS["mixtral_bf16"].with_(T=256, D=512, F=1024)
    inp = W.make_inputs(wl, device="cpu")
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"].to(DEV),
                     inp["w13"].to(DEV), inp["w2"].to(DEV), F=wl.F,
                     score=wl.score)
    x = inp["x"].to(DEV)
    replay = layer.capture(x, train=True)
    g = torch.Generator().manual_seed(9)
    dy = torch.randn(x.shape, generator=g).to(x.dtype).to(DEV)
    dx_graph = replay(dy).clone()
    dw2_graph = layer._train["dw2"].clone()
    layer.forward_train(x)
    dx_eager, _, _, dw2_eager = layer.backward(dy)
    torch.cuda.synchronize()
    assert torch.equal(dx_graph, dx_eager)
    assert torch.equal(dw2_graph, dw2_eager)
