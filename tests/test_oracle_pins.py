"""Pins for the CPU oracle: each test checks it against something other than
itself -- values the pages print, closed forms, brute-force enumeration,
invariants the method fixes, or an independent library routine.  The
mutation tests at the end plant plausible mistakes in the oracle and check
that at least one pin catches each."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle.moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- layout --
def test_worked_example_send_counts():
    g = _golden("dispatch_worked_example.json")
    idx = np.array(g["expert_indices"], dtype=np.int32)
    lay = O.dispatch_layout(idx, g["num_experts"], g["world_size"])
    assert lay["rank_send_counts"].tolist() == g["printed_send_counts"]
    # rows bound for each device, as sets, equal the page's device groups
    displs = lay["rank_send_displs"].tolist() + [lay["n_kept"]]
    for r, expect in enumerate(g["device_pair_sets"]):
        seg = lay["src_pair"][displs[r]:displs[r + 1]]
        assert sorted(seg.tolist()) == sorted(expect)
    assert lay["dropped"] == 0


def test_page_dispatch_matrix_invariants():
    g = _golden("dispatch_matrix_simulation.json")
    m = np.array(g["printed_matrix"])
    n, tpd, k = g["num_devices"], g["tokens_per_device"], g["top_k"]
    assert m.sum() == g["printed_total_pairs"] == n * tpd * k
    assert (m.sum(axis=1) == g["printed_expected_per_device"]).all()
    # the oracle's matrix on the same routing shape keeps those invariants,
    # and its column sums equal the rank send counts of the whole batch
    rng = np.random.default_rng(7)
    idx = rng.integers(0, g["num_experts"], size=(n * tpd, k))
    mo = O.dispatch_matrix(idx, n, n, g["num_experts"])
    assert (mo.sum(axis=1) == tpd * k).all() and mo.sum() == n * tpd * k
    lay = O.dispatch_layout(idx, g["num_experts"], n)
    assert (mo.sum(axis=0) == lay["rank_send_counts"]).all()
    # uniform routing: every entry near tpd*k/n (the page's entries lie
    # within about 15% of 256)
    assert np.abs(mo - tpd * k / n).max() < 0.25 * tpd * k / n


def _layout_brute(idx, E, R, cap):
    """The layout from its definition, by O(P^2) counting."""
    flat = np.asarray(idx).reshape(-1)
    P = len(flat)
    pos = [sum(1 for q in range(p) if flat[q] == flat[p]) for p in range(P)]
    kept = [cap is None or pos[p] < cap for p in range(P)]
    counts = [sum(1 for p in range(P) if kept[p] and flat[p] == e)
              for e in range(E)]
    offsets = [sum(counts[:e]) for e in range(E + 1)]
    dst = [offsets[flat[p]] + pos[p] if kept[p] else -1 for p in range(P)]
    epr = E // R
    rc = [sum(counts[r * epr:(r + 1) * epr]) for r in range(R)]
    return counts, offsets, dst, rc


@pytest.mark.parametrize("T,E,k,R,cap,distinct", [
    (13, 4, 2, 2, None, True), (13, 4, 2, 2, 3, True), (20, 6, 3, 3, 2, False),
    (9, 8, 1, 4, 1, False), (7, 3, 3, 1, 0, True), (1, 5, 2, 5, 1, True),
    (16, 4, 4, 2, 5, True)])
def test_layout_against_definition(T, E, k, R, cap, distinct):
    rng = np.random.default_rng(T * 31 + E)
    if distinct:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    else:
        idx = rng.integers(0, E, size=(T, k))
    lay = O.dispatch_layout(idx, E, R, cap)
    c = None if cap is None or cap <= 0 else cap
    counts, offsets, dst, rc = _layout_brute(idx, E, R, c)
    assert lay["counts"].tolist() == counts
    assert lay["offsets"].tolist() == offsets
    assert lay["dst_row"].tolist() == dst
    assert lay["rank_send_counts"].tolist() == rc
    assert lay["rank_send_displs"].tolist() == [sum(rc[:r]) for r in range(R)]
    # every kept pair appears exactly once; counts sum to P - dropped
    kept = [p for p in range(T * k) if dst[p] >= 0]
    assert sorted(lay["src_pair"].tolist()) == kept
    assert lay["counts"].sum() == T * k - lay["dropped"] == lay["n_kept"]
    assert lay["rank_send_counts"].sum() == lay["n_kept"]
    for r, p in enumerate(lay["src_pair"]):
        assert lay["dst_row"][p] == r
    # stable: within an expert, pair ids ascend
    for e in range(E):
        seg = lay["src_pair"][offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()


def test_capacity_values():
    # the two capacity-factor workloads print their capacities
    assert O.expert_capacity(1.25, 256, 2, 8) == 80
    assert O.expert_capacity(1.0, 16384, 1, 64) == 256
    assert O.expert_capacity(1.1, 100, 2, 8) == 28      # ceil(27.5)
    assert O.expert_capacity(1.5, 10, 1, 4) == 4        # ceil(3.75)
    assert O.expert_capacity(None, 10, 1, 4) is None


def test_infinite_capacity_equals_dropless():
    rng = np.random.default_rng(3)
    idx = rng.integers(0, 8, size=(200, 2))
    a = O.dispatch_layout(idx, 8, 4, None)
    b = O.dispatch_layout(idx, 8, 4, 10 ** 9)
    for key in ("counts", "offsets", "dst_row", "src_pair"):
        assert (a[key] == b[key]).all()


# ------------------------------------------------------------- selection --
def _brute_topk(keys, k, eligible):
    """The unique k-subset S of eligible experts such that every member
    beats every non-member (larger key, or equal key and lower index)."""
    def beats(i, j):
        return keys[i] > keys[j] or (keys[i] == keys[j] and i < j)
    winners = [S for S in itertools.combinations(eligible, k)
               if all(beats(i, j) for i in S for j in eligible if j not in S)]
    assert len(winners) == 1
    S = list(winners[0])
    order = sorted(S, key=lambda i: sum(1 for j in S if beats(j, i)))
    return order


@pytest.mark.parametrize("E,k,seed", [(5, 2, 0), (6, 3, 1), (8, 1, 2),
                                      (4, 4, 3), (7, 2, 4)])
def test_topk_brute_force_with_ties(E, k, seed):
    rng = np.random.default_rng(seed)
    logits = rng.integers(-2, 3, size=(40, E)).astype(np.float32)
    logits[0] = 0.0
    logits[1, :] = -0.0
    idx, _ = O.route_from_logits(logits, k, O.SOFTMAX_TOPK)
    for t in range(40):
        assert idx[t].tolist() == _brute_topk(logits[t], k, list(range(E)))


def test_group_limited_brute_force():
    rng = np.random.default_rng(11)
    E, G, TG, k, gk = 16, 4, 2, 3, 2
    gs = E // G
    for t in range(60):
        logits = rng.integers(-3, 4, size=(1, E)).astype(np.float32) * 0.5
        bias = rng.integers(-1, 2, size=E).astype(np.float32) * 0.125
        idx, _ = O.route_from_logits(logits, k, O.SIGMOID_BIAS, bias,
                                     n_groups=G, topk_groups=TG,
                                     group_score_topk=gk)
        s = scipy.special.expit(logits[0].astype(np.float64)).astype(np.float32)
        keys = (s + bias).astype(np.float32)
        # group score: the best sum of any gk keys in the group, in fp32
        # (order-free for two terms)
        score = []
        for g in range(G):
            mem = range(g * gs, (g + 1) * gs)
            score.append(max(np.float32(keys[a] + keys[b]) for a, b in
                             itertools.combinations(mem, 2)))
        groups = _brute_topk(np.array(score), TG, list(range(G)))
        eligible = sorted(e for g in groups for e in range(g * gs, (g + 1) * gs))
        assert idx[0].tolist() == _brute_topk(keys, k, eligible)


def _sigmoid_grid():
    # dense grid over [-95, 95] (past both ends of fp32's useful range),
    # random points, and the special values
    return np.concatenate([np.linspace(-95, 95, 400001),
                           np.random.default_rng(1).standard_normal(200000) * 4,
                           [0.0, -0.0, 1e-30, -1e-30, 87.0, -87.0, 88.0,
                            -88.0, 103.0, -103.0]]).astype(np.float32)


def test_sigmoid_key_is_expit_rounded_once():
    # the selection score fp32(sigmoid(l)) against scipy's float64 expit
    # rounded once, bit for bit, over the whole range
    l = _sigmoid_grid()
    got = O.sigmoid_f32(l)
    ref = scipy.special.expit(l.astype(np.float64)).astype(np.float32)
    assert got.dtype == np.float32
    assert (got.view(np.uint32) == ref.view(np.uint32)).all()
    # closed forms: sigmoid(0) = 1/2 exactly, saturation at the ends
    assert O.sigmoid_f32(np.float32([0.0, -0.0])).tolist() == [0.5, 0.5]
    assert O.sigmoid_f32(np.float32([95.0]))[0] == 1.0
    assert 0.0 < O.sigmoid_f32(np.float32([-95.0]))[0] < 1e-41
    # monotone non-decreasing on the sorted grid
    g = O.sigmoid_f32(np.sort(l))
    assert (np.diff(g.astype(np.float64)) >= 0).all()


def test_sigmoid_key_correctly_rounded():
    # 50-digit evaluation of 1/(1+e^-l) rounded to the nearest fp32 value:
    # the oracle's score is the correctly rounded sigmoid on a sample
    # spanning the range (a float64 evaluation can differ only within a
    # few float64 ulp of an fp32 rounding boundary)
    import mpmath
    mpmath.mp.dps = 50
    rng = np.random.default_rng(5)
    l = np.concatenate([rng.uniform(-90, 90, 1500), rng.standard_normal(1500)]
                       ).astype(np.float32)
    got = O.sigmoid_f32(l)
    for li, gi in zip(l.tolist(), got.tolist()):
        exact = 1 / (1 + mpmath.exp(-mpmath.mpf(li)))
        lo = np.float32(float(exact))
        # the two fp32 neighbours around the exact value; the nearer wins
        cands = [lo, np.nextafter(lo, np.float32(-1)), np.nextafter(lo, np.float32(2))]
        best = min(cands, key=lambda c: abs(mpmath.mpf(float(c)) - exact))
        assert gi == float(best), (li, gi, float(best))


def test_sigmoid_bias_selects_but_does_not_weight():
    logits = np.array([[0.0, 0.5, 1.0, -1.0]], dtype=np.float32)
    bias = np.array([0.0, 0.0, 0.0, 5.0], dtype=np.float32)
    idx, gate = O.route_from_logits(logits, 2, O.SIGMOID_BIAS, bias)
    assert idx[0].tolist() == [3, 2]
    s = scipy.special.expit(np.array([-1.0, 1.0]))
    np.testing.assert_allclose(gate[0], s / s.sum(), rtol=1e-14)


# ----------------------------------------------------------------- gates --
def test_gates_match_library_softmax():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 8)).astype(np.float32)
    idx, g = O.route_from_logits(logits, 2, O.SOFTMAX_TOPK)
    for t in range(50):
        ref = scipy.special.softmax(logits[t, idx[t]].astype(np.float64))
        np.testing.assert_allclose(g[t], ref, rtol=1e-13)
    idx, g = O.route_from_logits(logits, 1, O.SOFTMAX_FULL)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert (idx[:, 0] == np.argmax(logits, axis=1)).all()
    np.testing.assert_allclose(g[:, 0], p.max(axis=1), rtol=1e-13)
    # k = 1 with the top-k softmax: every gate is exactly one
    _, g1 = O.route_from_logits(logits, 1, O.SOFTMAX_TOPK)
    assert (g1 == 1.0).all()


def test_router_logits_exact_on_integers():
    rng = np.random.default_rng(2)
    x = rng.integers(-8, 9, size=(5, 12)).astype(np.float32)
    w = rng.integers(-8, 9, size=(3, 12)).astype(np.float32)
    off = np.array([0.5, -1.0, 2.0], dtype=np.float32)
    got = O.router_logits(x, w, off)
    for t in range(5):
        for e in range(3):
            exact = sum(int(x[t, d]) * int(w[e, d]) for d in range(12))
            assert got[t, e] == np.float32(exact + float(off[e]))


# --------------------------------------------------------------- experts --
def _torch_swiglu(h, w1, w3, w2):
    h = torch.as_tensor(h, dtype=torch.float64)
    a = torch.nn.functional.silu(h @ torch.as_tensor(w1).double().T)
    b = h @ torch.as_tensor(w3).double().T
    return ((a * b) @ torch.as_tensor(w2).double().T).numpy()


def test_single_expert_equals_plain_swiglu_mlp():
    rng = np.random.default_rng(9)
    T, D, F = 17, 12, 20
    x = rng.standard_normal((T, D))
    w13 = rng.standard_normal((1, 2 * F, D)) * 0.3
    w2 = rng.standard_normal((1, D, F)) * 0.3
    w_r = rng.standard_normal((1, D))
    out = O.moe_forward(x, w_r, k=1, E=1, R=1, mode=O.SOFTMAX_TOPK,
                        w13=w13, w2=w2)
    ref = _torch_swiglu(x, w13[0, :F], w13[0, F:], w2[0])
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_k_equals_E_is_dense_mixture():
    rng = np.random.default_rng(10)
    T, D, F, E = 9, 8, 6, 4
    x = rng.standard_normal((T, D))
    w_r = rng.standard_normal((E, D))
    w13 = rng.standard_normal((E, 2 * F, D)) * 0.3
    w2 = rng.standard_normal((E, D, F)) * 0.3
    out = O.moe_forward(x, w_r, k=E, E=E, R=2, mode=O.SOFTMAX_TOPK,
                        w13=w13, w2=w2)
    logits = (torch.as_tensor(x) @ torch.as_tensor(w_r).T).float().double()
    p = torch.softmax(logits, dim=1).numpy()
    ref = sum(p[:, [e]] * _torch_swiglu(x, w13[e, :F], w13[e, F:], w2[e])
              for e in range(E))
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-12)


def test_identity_experts_reproduce_x():
    rng = np.random.default_rng(4)
    T, D, E = 64, 16, 8
    x = rng.standard_normal((T, D))
    w_r = rng.standard_normal((E, D))
    for mode, k in ((O.SOFTMAX_TOPK, 2), (O.SIGMOID_BIAS, 3),
                    (O.SOFTMAX_TOPK, 1)):
        out = O.moe_forward(x, w_r, k=k, E=E, R=4, mode=mode)
        np.testing.assert_allclose(out["y"], x, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(out["topk_gate"].sum(1), 1.0, rtol=1e-14)


def test_dropped_pairs_contribute_zero():
    # every token routed to expert 0 with capacity 2: only tokens 0 and 1
    # keep their pair; the others' outputs are exactly zero
    T, D = 6, 4
    x = np.arange(T * D, dtype=np.float64).reshape(T, D) + 1.0
    idx = np.zeros((T, 1), dtype=np.int32)
    gate = np.ones((T, 1))
    out = O.moe_forward(x, None, k=1, E=2, R=1, mode=O.SOFTMAX_TOPK,
                        capacity=2, topk_idx=idx, topk_gate=gate)
    assert out["dst_row"].tolist() == [0, 1, -1, -1, -1, -1]
    np.testing.assert_array_equal(out["y"][:2], x[:2])
    assert (out["y"][2:] == 0).all()


def test_volume_equals_two_TKD():
    rng = np.random.default_rng(6)
    T, D, E, k = 40, 8, 8, 3
    x = rng.standard_normal((T, D))
    w_r = rng.standard_normal((E, D))
    out = O.moe_forward(x, w_r, k=k, E=E, R=4, mode=O.SOFTMAX_TOPK)
    moved = out["xp"].size + sum(
        D for p in range(T * k) if out["dst_row"][p] >= 0)
    assert moved == O.dispatch_combine_volume(T, k, D) == 2 * T * k * D
    # per-rank dispatch volume formula: (EP-1)/EP of T*k*D elements cross
    assert O.dispatch_bytes_per_rank(T, k, D, 4, 2) == \
        T * k * D * 2 * 3 / 4


def test_token_output_matches_forward():
    rng = np.random.default_rng(12)
    T, D, F, E, k = 20, 8, 6, 4, 2
    x = rng.standard_normal((T, D))
    w_r = rng.standard_normal((E, D))
    w13 = rng.standard_normal((E, 2 * F, D)) * 0.3
    w2 = rng.standard_normal((E, D, F)) * 0.3
    out = O.moe_forward(x, w_r, k=k, E=E, R=2, mode=O.SOFTMAX_TOPK,
                        w13=w13, w2=w2, capacity=6)

    def ew(e):
        return w13[e, :F], w13[e, F:], w2[e]
    for t in range(T):
        yt = O.token_output(x[t], t, out["topk_idx"], out["topk_gate"],
                            out["dst_row"], k, ew)
        np.testing.assert_allclose(yt, out["y"][t], rtol=1e-12, atol=1e-14)


# ------------------------------------------------- planted mistakes -------
def _run_pins(funcs):
    failed = 0
    for f in funcs:
        try:
            f()
        except AssertionError:
            failed += 1
    return failed


def test_mutation_swapped_gate_and_up_is_caught(monkeypatch):
    monkeypatch.setattr(O, "split_w13", lambda w: (w[w.shape[0] // 2:],
                                                   w[:w.shape[0] // 2]))
    assert _run_pins([test_single_expert_equals_plain_swiglu_mlp]) == 1


def test_mutation_silu_sign_is_caught(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda z: z / (1.0 + np.exp(z)))
    assert _run_pins([test_single_expert_equals_plain_swiglu_mlp,
                      test_k_equals_E_is_dense_mixture]) == 2


def test_mutation_tie_break_is_caught(monkeypatch):
    monkeypatch.setattr(O, "_order_desc",
                        lambda v, ids: sorted(ids, key=lambda i: (-float(v[i]), -i)))
    assert _run_pins([lambda: test_topk_brute_force_with_ties(5, 2, 0)]) == 1


def test_mutation_unstable_layout_is_caught(monkeypatch):
    real = O.dispatch_layout

    def reversed_order(idx, E, R, capacity=None):
        flat = np.asarray(idx).reshape(-1)
        lay = real(flat[::-1].copy(), E, R, capacity)
        return lay
    monkeypatch.setattr(O, "dispatch_layout", reversed_order)
    assert _run_pins([lambda: test_layout_against_definition(
        13, 4, 2, 2, 3, True)]) == 1


def test_mutation_dropped_gate_is_caught(monkeypatch):
    real = O.combine

    def no_gate(yp, dst_row, gate, T, k):
        return real(yp, dst_row, np.ones_like(gate), T, k)
    monkeypatch.setattr(O, "combine", no_gate)
    assert _run_pins([test_identity_experts_reproduce_x,
                      test_k_equals_E_is_dense_mixture]) == 2
