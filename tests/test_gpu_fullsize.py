"""Parity at the full workload sizes, in the launch configuration bench.py
times (same layer construction, same seeded device inputs).

At these sizes the oracle checks, on every token:
  * router logits within the fp32-accumulation bound, and top-k ids
    bit-exact from the logits the kernel used, gates within 2e-6;
  * the layout bit-exact (counts, offsets, dst_row, src_pair, rank counts);
  * the permute as a pure copy (every kept buffer row equals its token row);
on every expert that received rows, the grouped FFN's output rows at the
first, middle and last row of its segment against the oracle's float64
SwiGLU expert at the full D x F contraction (max|yp - ref| / max|ref| over
the expert's checked rows <= 1e-2, bf16);
and, on a seeded sample of tokens, the layer output from the layer equation
itself (max|y - y_ref| / max|y_ref| <= 1e-2).  The expert references are
computed one expert at a time, so host memory holds one expert's float64
weights at a time.  Identity-expert sweeps also check y against x on every
token.
"""
import numpy as np
import pytest
import torch

import bench
import oracle.moe_oracle as O
from combine_router_gemm_top_b300 import workloads as W

pytestmark = pytest.mark.gpu

SAMPLE_TOKENS = {"mixtral_bf16": 64, "deepseek_bf16": 64, "switch_bf16": 64}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, ref):
    den = np.abs(ref).max()
    return np.abs(got - ref).max() / (den if den > 0 else 1.0)


def run_full(name):
    wl = W.WORKLOADS[name]
    dev = torch.device("cuda", 0)
    layer, inp = bench.build_layer(wl, dev, wl.seed)
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
    layer.logits = logits
    x = inp["x"]
    idx_in, gate_in = inp.get("topk_idx"), inp.get("topk_gate")
    layer.route(x)
    layer.dispatch_layout(idx_in)
    layer.permute(x)
    layer.grouped_ffn()
    y = layer.combine(gate_in)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    return wl, layer, inp, y


def check_route(wl, layer, inp):
    x64, w64 = f64(inp["x"]), f64(inp["w_r"])
    lg = layer.logits.cpu().numpy()
    off = None if inp["logit_offset"] is None else \
        inp["logit_offset"].cpu().numpy()
    ref_l = O.router_logits(x64, w64, off)
    bound = 2.0 ** -16 * (np.abs(x64) @ np.abs(w64).T) + 1e-6
    assert (np.abs(lg.astype(np.float64) - ref_l) <= bound).all()
    bias = None if inp["sel_bias"] is None else inp["sel_bias"].cpu().numpy()
    ridx, rgate = O.route_from_logits(lg, wl.k, wl.score, bias, wl.n_groups,
                                      wl.topk_groups, wl.group_score_topk)
    assert (layer.topk_idx.cpu().numpy() == ridx).all()
    assert np.abs(f64(layer.topk_gate) - rgate).max() <= 2e-6
    return ridx


def check_layout_and_permute(wl, layer, idx, x):
    cap = O.expert_capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    ref = O.dispatch_layout(idx, wl.E, wl.R, cap)
    P = wl.T * wl.k
    assert layer.expert_counts.cpu().numpy().tolist() == ref["counts"].tolist()
    assert layer.expert_offsets.cpu().numpy().tolist() == \
        ref["offsets"].tolist()
    dst = layer.dst_row.cpu().numpy()[:P]
    assert dst.tolist() == ref["dst_row"].tolist()
    n = ref["n_kept"]
    assert layer.src_pair.cpu().numpy()[:n].tolist() == ref["src_pair"].tolist()
    assert layer.rank_send_counts.cpu().numpy().tolist() == \
        ref["rank_send_counts"].tolist()
    assert layer.rank_send_displs.cpu().numpy().tolist() == \
        ref["rank_send_displs"].tolist()
    assert int(layer.n_kept.item()) == n
    assert int(layer.n_dropped.item()) == P - n
    # permute: a pure copy of each kept pair's token row
    d = torch.as_tensor(dst, device=x.device, dtype=torch.int64)
    kept = d >= 0
    pairs = torch.arange(P, device=x.device)[kept]
    assert torch.equal(layer.xp[d[kept]], x[pairs // wl.k])
    return ref


def expert_references(wl, inp, rows_by_expert, token_of_row):
    """Float64 SwiGLU outputs of the requested buffer rows, expert by
    expert: {row: yp_ref[row]} for rows_by_expert = {e: [rows]}, each row's
    input being its token's x row."""
    F = wl.F
    out = {}
    for e in sorted(rows_by_expert):
        rows = sorted(set(rows_by_expert[e]))
        w13 = inp["w13"][e].to("cpu").to(torch.float64).numpy()
        w2 = inp["w2"][e].to("cpu").to(torch.float64).numpy()
        toks = torch.as_tensor([token_of_row[r] for r in rows])
        h = inp["x"][toks.to(inp["x"].device)].to("cpu").to(
            torch.float64).numpy()
        ref = O.swiglu_expert(h, w13[:F], w13[F:], w2)
        for r, v in zip(rows, ref):
            out[r] = v
        del w13, w2
    return out


@pytest.mark.parametrize("name", ["mixtral_bf16", "deepseek_bf16",
                                  "switch_bf16"])
def test_fullsize_layer(name):
    wl, layer, inp, y = run_full(name)
    idx = check_route(wl, layer, inp)
    ref = check_layout_and_permute(wl, layer, idx, inp["x"])
    k = wl.k
    off = ref["offsets"]
    src_pair = ref["src_pair"]
    token_of_row = {int(r): int(p) // k for r, p in enumerate(src_pair)}
    # every expert with rows: the first, middle and last row of its segment
    seg_rows = {}
    for e in range(wl.E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            seg_rows[e] = [a, a + (b - a) // 2, b - 1]
    # sampled tokens: every kept slot's row
    g = np.random.default_rng(wl.seed)
    toks = np.sort(g.choice(wl.T, SAMPLE_TOKENS[name], replace=False))
    want = {e: list(v) for e, v in seg_rows.items()}
    for t in toks:
        for j in range(k):
            r = int(ref["dst_row"][t * k + j])
            if r >= 0:
                want.setdefault(int(idx[t][j]), []).append(r)
    yp_ref = expert_references(wl, inp, want, token_of_row)
    yp = layer.yp
    assert len(seg_rows) == int((ref["counts"] > 0).sum())
    for e, rows in seg_rows.items():
        got = f64(yp[torch.as_tensor(rows, device=yp.device)])
        r64 = np.stack([yp_ref[r] for r in rows])
        assert np.isfinite(got).all(), e
        assert rel_err(got, r64) <= 1e-2, (e, rel_err(got, r64))
    # the layer equation on the sampled tokens, from the same references
    gate = f64(layer.topk_gate)
    ref_rows = np.zeros((len(toks), wl.D))
    for i, t in enumerate(toks):
        for j in range(k):
            r = int(ref["dst_row"][t * k + j])
            if r >= 0:
                ref_rows[i] += gate[t, j] * yp_ref[r]
    got = f64(y[torch.as_tensor(toks, device=y.device)])
    assert np.isfinite(got).all()
    assert rel_err(got, ref_rows) <= 1e-2


@pytest.mark.parametrize("T", [4096, 16384, 65536])
@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_fullsize_sweep(T, routing):
    name = f"sweep_bf16_{routing}_T{T}"
    wl, layer, inp, y = run_full(name)
    if T == 65536:
        check_route(wl, layer, inp)      # the router timed in the sweep
    idx = inp["topk_idx"].cpu().numpy()
    ref = check_layout_and_permute(wl, layer, idx, inp["x"])
    # identity experts and Dirichlet gates: y = sum_j g_j x = x, every token
    xf, yf = inp["x"].float(), y.float()
    assert float((yf - xf).abs().max()) <= 1e-2 * float(xf.abs().max())
    # and the combine itself against the oracle on sampled tokens
    toks = np.arange(0, T, T // 64)
    gate = f64(inp["topk_gate"])
    ref_rows = np.stack([O.token_output(f64(inp["x"][t]), t, idx, gate,
                                        ref["dst_row"], wl.k, lambda e: None)
                         for t in toks])
    assert rel_err(f64(y[torch.as_tensor(toks, device=y.device)]),
                   ref_rows) <= 1e-2
