"""Pins for the oracle's backward pass: central finite differences of the
oracle's own forward (an independent route to every gradient), torch
autograd in float64 on a plain torch restatement of the layer with the
routing held fixed, closed forms, the page's backward volume, and planted
mistakes that a pin must catch."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O


def _case(seed, T=4, D=6, E=4, k=2, F=5, scale=0.7):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, D))
    w_r = rng.normal(size=(E, D)) * scale
    w13 = rng.normal(size=(E, 2 * F, D)) * 0.5
    w2 = rng.normal(size=(E, D, F)) * 0.5
    dy = rng.normal(size=(T, D))
    return x, w_r, w13, w2, dy


def _loss(x, w_r, w13, w2, dy, k, E, mode, **kw):
    y = O.moe_forward(x, w_r, k, E, 1, mode, w13=w13, w2=w2, **kw)
    return float(np.sum(dy * y["y"])), y["topk_idx"], y["dst_row"]


def _fd_check(x, w_r, w13, w2, dy, k, E, mode, h=1e-3, tol=2e-3, **kw):
    """Central differences of L = sum(dy * y).  The oracle rounds router
    logits to fp32 (as the kernel does), which adds noise of about
    |dL/dl| * 1e-7 / h to each quotient; h = 1e-3 keeps that and the
    O(h^2) truncation near 1e-5 relative, far below what a wrong formula
    gives."""
    g = O.moe_backward(x, w_r, dy, k, E, 1, mode, w13=w13, w2=w2, **kw)
    _, idx0, dst0 = _loss(x, w_r, w13, w2, dy, k, E, mode, **kw)
    params = dict(x=x, w_r=w_r, w13=w13, w2=w2)
    grads = dict(x=g["dx"], w_r=g["dw_r"], w13=g["dw13"], w2=g["dw2"])
    for name, arr in params.items():
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            vals = []
            for s in (+h, -h):
                arr[i] = old + s
                L, idx, dst = _loss(x, w_r, w13, w2, dy, k, E, mode, **kw)
                # the perturbation must not move the routing decision
                assert (idx == idx0).all() and (dst == dst0).all()
                vals.append(L)
            arr[i] = old
            num[i] = (vals[0] - vals[1]) / (2 * h)
        err = np.abs(num - grads[name]).max()
        assert err <= tol * max(1.0, np.abs(num).max()), (name, err)
    return g


@pytest.mark.parametrize("mode,k,seed", [
    (O.SOFTMAX_TOPK, 2, 0), (O.SOFTMAX_TOPK, 3, 1),
    (O.SOFTMAX_FULL, 1, 2), (O.SIGMOID_BIAS, 2, 3)])
def test_gradients_match_finite_differences(mode, k, seed):
    x, w_r, w13, w2, dy = _case(seed)
    kw = {}
    if mode == O.SIGMOID_BIAS:
        kw["sel_bias"] = np.array([0.05, -0.02, 0.0, 0.03], np.float32)
    _fd_check(x, w_r, w13, w2, dy, k, 4, mode, **kw)


def test_dropped_pairs_have_no_gradient_path():
    # capacity 1 with 6 tokens on 3 experts: most pairs drop; their gates
    # get zero gradient and their experts see nothing from them
    x, w_r, w13, w2, dy = _case(7, T=6, E=3)
    g = _fd_check(x, w_r, w13, w2, dy, 2, 3, O.SOFTMAX_TOPK, capacity=1)
    dropped = g["forward"]["dst_row"].reshape(6, 2) < 0
    assert dropped.any()
    assert (g["dgate"][dropped] == 0).all()


def _torch_layer(x, w_r, w13, w2, idx, keep, mode):
    """The layer equation in float64 torch with the selection fixed."""
    l = x @ w_r.T
    T, k = idx.shape
    F = w13.shape[1] // 2
    y = torch.zeros_like(x)
    for t in range(T):
        sel = idx[t]
        if mode == O.SOFTMAX_TOPK:
            g = torch.softmax(l[t, sel], 0)
        elif mode == O.SOFTMAX_FULL:
            g = torch.softmax(l[t], 0)[sel]
        else:
            s = torch.sigmoid(l[t, sel])
            g = s / s.sum()
        for j in range(k):
            if not keep[t, j]:
                continue
            e = int(sel[j])
            h = x[t]
            a = torch.nn.functional.silu(w13[e, :F] @ h) * (w13[e, F:] @ h)
            y[t] = y[t] + g[j] * (w2[e] @ a)
    return y


@pytest.mark.parametrize("mode,k", [(O.SOFTMAX_TOPK, 2),
                                    (O.SOFTMAX_FULL, 1),
                                    (O.SIGMOID_BIAS, 3)])
def test_gradients_match_torch_autograd(mode, k):
    x, w_r, w13, w2, dy = _case(11, T=16, D=8, E=5, F=6)
    g = O.moe_backward(x, w_r, dy, k, 5, 1, mode, w13=w13, w2=w2,
                       capacity=5)
    fw = g["forward"]
    idx = torch.tensor(fw["topk_idx"].astype(np.int64))
    keep = torch.tensor((fw["dst_row"] >= 0).reshape(16, k))
    tx, tr, t13, t2 = (torch.tensor(a, requires_grad=True)
                       for a in (x, w_r, w13, w2))
    y = _torch_layer(tx, tr, t13, t2, idx, keep, mode)
    (y * torch.tensor(dy)).sum().backward()
    # torch differentiates the unrounded logits, the oracle rounds them to
    # fp32 first (as the kernel does): agreement to ~1e-7 relative
    for ours, ref in ((g["dx"], tx.grad), (g["dw_r"], tr.grad),
                      (g["dw13"], t13.grad), (g["dw2"], t2.grad)):
        r = ref.numpy()
        assert np.abs(ours - r).max() <= 1e-6 * np.abs(r).max()


def test_identity_top1_passes_dy_through():
    # identity experts and a single softmax_topk slot: the gate is 1 for
    # every logit value, so dx = dy exactly and the router gets nothing
    rng = np.random.default_rng(5)
    T, D, E = 9, 4, 3
    x = rng.normal(size=(T, D))
    w_r = rng.normal(size=(E, D))
    dy = rng.normal(size=(T, D))
    g = O.moe_backward(x, w_r, dy, 1, E, 1, O.SOFTMAX_TOPK)
    np.testing.assert_allclose(g["dx"], dy, rtol=0, atol=1e-15)
    assert np.abs(g["dw_r"]).max() == 0.0


def test_backward_volume_mirrors_forward():
    # the pages' Volume_total = 4*B*S*k*H elements per layer (forward and
    # backward each dispatch and combine T*k rows of D)
    rng = np.random.default_rng(2)
    T, D, E, k = 12, 5, 4, 2
    x = rng.normal(size=(T, D))
    w_r = rng.normal(size=(E, D))
    g = O.moe_backward(x, w_r, rng.normal(size=(T, D)), k, E, 1,
                       O.SOFTMAX_TOPK)
    fw = g["forward"]
    moved = (fw["xp"].size + fw["yp"].size          # forward dispatch/combine
             + g["dyp"].size + g["dxp"].size)       # backward mirror
    assert moved == 4 * T * k * D == 2 * O.dispatch_combine_volume(T, k, D)


# ------------------------------------------------- planted mistakes -------
def _fails(f):
    try:
        f()
    except AssertionError:
        return True
    return False


def test_mutation_silu_grad_is_caught(monkeypatch):
    monkeypatch.setattr(O, "silu_grad", lambda z: 1.0 / (1.0 + np.exp(-z)))
    assert _fails(lambda: test_gradients_match_finite_differences(
        O.SOFTMAX_TOPK, 2, 0))


def test_mutation_sigmoid_gate_norm_is_caught(monkeypatch):
    real = O.gate_backward

    def no_norm(l, sel, dgate, mode):
        if mode != O.SIGMOID_BIAS:
            return real(l, sel, dgate, mode)
        s = O.sigmoid_f64(np.asarray(l, np.float64)[list(sel)])
        dl = np.zeros(len(l))
        dl[list(sel)] = np.asarray(dgate) * s * (1.0 - s)
        return dl
    monkeypatch.setattr(O, "gate_backward", no_norm)
    assert _fails(lambda: test_gradients_match_torch_autograd(
        O.SIGMOID_BIAS, 3))


def test_mutation_ungated_dispatch_is_caught(monkeypatch):
    # the backward dispatches dy without the gate factor (its forward pass
    # reports unit gates): the autograd pin must catch it
    orig_forward = O.moe_forward

    def fwd_gate_one(*a, **kw):
        out = orig_forward(*a, **kw)
        out["topk_gate"] = np.ones_like(out["topk_gate"])
        return out
    monkeypatch.setattr(O, "moe_forward", fwd_gate_one)
    assert _fails(lambda: test_gradients_match_torch_autograd(
        O.SOFTMAX_TOPK, 2))
