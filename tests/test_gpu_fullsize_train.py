"""Parity of the training step at the full Mixtral-like and DeepSeek-like
sizes, in the configuration `bench.py --train` times (same layer
construction, seeded device inputs, forward on the 64-row aligned layout,
then the backward pass).

What the oracle checks at these sizes:
  * dx on a seeded sample of tokens, from the chain rule of the layer
    equation token by token: the expert backward of each kept slot with
    the gate-scaled dy, plus the router term (dlogits from the oracle's
    gate backward, times W_r);
  * dW13 and dW2 of one whole expert (the smallest non-empty one) in
    float64 from that expert's rows;
  * dW_r in full (the oracle's dlogits^T x over every token).
Bar: max|g - g_ref| / max|g_ref| <= 2e-2 (dH, [dG|dU] and H are bf16 between
the GEMMs, as H is in the forward).
"""
import numpy as np
import pytest
import torch

import bench
import oracle.moe_oracle as O
from combine_router_gemm_top_b300 import workloads as W

pytestmark = pytest.mark.gpu

SAMPLE = {"mixtral_bf16": 8, "deepseek_bf16": 4}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel(got, ref):
    den = np.abs(ref).max()
    return np.abs(np.asarray(got) - ref).max() / (den if den > 0 else 1.0)


@pytest.mark.parametrize("name", ["mixtral_bf16", "deepseek_bf16"])
def test_training_step_full_size(name):
    wl = W.WORKLOADS[name]
    dev = torch.device("cuda", 0)
    layer, inp = bench.build_layer(wl, dev, wl.seed)
    x = inp["x"]
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 17)
    dy = torch.randn(x.shape, generator=g, device=dev).to(x.dtype)
    layer.forward_train(x)
    dx, dw_r, dw13, dw2 = layer.backward(dy)
    torch.cuda.synchronize()
    assert layer.device_status() == 0

    k, E, F, D = wl.k, wl.E, wl.F, wl.D
    logits = layer.logits.cpu().numpy()
    idx = layer.topk_idx.cpu().numpy()
    gate = f64(layer.topk_gate)
    dst = layer.dst_row.cpu().numpy()
    X, DY, WR = f64(x), f64(dy), f64(inp["w_r"])
    # routing decision equals the oracle's on the kernel's logits
    ridx, rgate = O.route_from_logits(
        logits, k, wl.score,
        None if inp["sel_bias"] is None else inp["sel_bias"].cpu().numpy(),
        wl.n_groups, wl.topk_groups, wl.group_score_topk)
    assert (idx == ridx).all()

    def expert_w(e):
        w13 = f64(inp["w13"][e])
        return w13[:F], w13[F:], f64(inp["w2"][e])

    # expert outputs of the sampled tokens from the layer equation
    rng = np.random.default_rng(0)
    sample = rng.choice(wl.T, SAMPLE[name], replace=False)
    dlog = np.zeros((wl.T, E))
    yp_of = {}
    for t in sample:
        for j in range(k):
            if dst[t * k + j] >= 0:
                w1, w3, w2 = expert_w(int(idx[t, j]))
                yp_of[(t, j)] = O.swiglu_expert(X[t:t + 1], w1, w3, w2)[0]
    # dgate and dlogits for every token need each kept pair's expert output;
    # they take the device's forward rows, which the sample checks against
    # the layer equation
    b = layer._train
    ya = f64(b["ya"])
    dsta = b["dst_a"].cpu().numpy()
    for t in range(wl.T):
        dg = np.zeros(k)
        for j in range(k):
            r = dsta[t * k + j]
            if r >= 0:
                dg[j] = DY[t] @ ya[r]
        dlog[t] = O.gate_backward(logits[t], idx[t], dg, wl.score)
    for (t, j), yref in yp_of.items():
        assert rel(ya[dsta[t * k + j]], yref) <= 1e-2

    # dx on the sample
    dxg = f64(dx)
    for t in sample:
        ref = dlog[t] @ WR
        for j in range(k):
            if dst[t * k + j] < 0:
                continue
            w1, w3, w2 = expert_w(int(idx[t, j]))
            dh, _, _, _ = O.expert_backward(X[t:t + 1], w1, w3, w2,
                                            gate[t, j] * DY[t:t + 1])
            ref = ref + dh[0]
        assert rel(dxg[t], ref) <= 2e-2

    # dW_r over all tokens
    assert rel(f64(dw_r), dlog.T @ X) <= 2e-2

    # one whole expert's weight gradients
    counts = layer.expert_counts.cpu().numpy().astype(np.int64)
    e = int(np.argmin(np.where(counts > 0, counts, np.iinfo(np.int64).max)))
    pairs = [p for p in range(wl.T * k) if dst[p] >= 0 and idx.reshape(-1)[p] == e]
    rows = np.array([p // k for p in pairs])
    gts = np.array([gate.reshape(-1)[p] for p in pairs])
    w1, w3, w2 = expert_w(e)
    _, dw1, dw3, dw2e = O.expert_backward(X[rows], w1, w3, w2,
                                          gts[:, None] * DY[rows])
    assert rel(f64(dw13[e, :F]), dw1) <= 2e-2
    assert rel(f64(dw13[e, F:]), dw3) <= 2e-2
    assert rel(f64(dw2[e]), dw2e) <= 2e-2
