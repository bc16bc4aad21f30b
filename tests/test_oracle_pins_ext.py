"""Pins for the oracle's router statistics, bias update, dispatch matrix and
padded static-capacity layout: closed forms, hand-worked examples, library
routines and invariants, plus planted mistakes that a pin must catch."""
import numpy as np
import pytest
import scipy.special

import oracle.moe_oracle as O


# ------------------------------------------------------- router statistics
def _even_routing(T, k, E):
    """Token t takes experts (t*k + j) mod E: every expert gets T*k/E pairs
    when E divides T*k."""
    return np.array([[(t * k + j) % E for j in range(k)] for t in range(T)],
                    dtype=np.int32)


@pytest.mark.parametrize("mode", [O.SOFTMAX_TOPK, O.SOFTMAX_FULL,
                                  O.SIGMOID_BIAS])
@pytest.mark.parametrize("T,k,E", [(16, 2, 8), (12, 1, 4), (24, 8, 16)])
def test_aux_loss_is_alpha_at_perfect_balance(mode, T, k, E):
    # equal logits give P_i = 1/E, even routing gives f_i = 1/E, so
    # L_aux = alpha * E * E * (1/E)^2 = alpha
    st = O.router_stats(np.zeros((T, E), np.float32), _even_routing(T, k, E),
                        E, mode, alpha=0.01)
    assert st["aux_loss"] == pytest.approx(0.01, rel=1e-12)
    assert (st["counts_routed"] == T * k // E).all()


def test_aux_loss_collapse_approaches_alpha_times_E():
    # every token on expert 0 with probability ~1: f_0 = 1, P_0 -> 1
    T, E = 10, 8
    logits = np.zeros((T, E), np.float32)
    logits[:, 0] = 60.0
    idx = np.zeros((T, 1), np.int32)
    st = O.router_stats(logits, idx, E, O.SOFTMAX_FULL, alpha=1.0)
    assert st["f"][0] == 1.0
    assert st["aux_loss"] == pytest.approx(E, rel=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_router_stats_match_library_routines(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 37, 12, 3
    logits = rng.normal(size=(T, E)).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    st = O.router_stats(logits, idx, E, O.SOFTMAX_TOPK, alpha=0.5)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1).mean(0)
    f = np.bincount(idx.reshape(-1), minlength=E) / (T * k)
    np.testing.assert_allclose(st["P"], p, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(st["f"], f)
    assert st["aux_loss"] == pytest.approx(0.5 * E * float(f @ p), rel=1e-13)
    s = scipy.special.expit(logits.astype(np.float64))
    ps = (s / s.sum(1, keepdims=True)).mean(0)
    st2 = O.router_stats(logits, idx, E, O.SIGMOID_BIAS, alpha=0.5)
    np.testing.assert_allclose(st2["P"], ps, rtol=1e-13, atol=1e-15)
    for s_ in (st, st2):
        assert s_["f"].sum() == pytest.approx(1.0, abs=1e-15)
        assert s_["P"].sum() == pytest.approx(1.0, abs=1e-12)


def test_bias_update_hand_example():
    # E=4, T=4, k=2: loads [4, 2, 2, 0] against the mean 2 -> the
    # overloaded expert is lowered, the idle one raised, the rest kept
    b = O.bias_update(np.array([0.1, -0.2, 0.0, 0.3], np.float32),
                      np.array([4, 2, 2, 0]), T=4, k=2, gamma=0.25)
    np.testing.assert_array_equal(
        b, np.array([0.1 - 0.25, -0.2, 0.0, 0.3 + 0.25], np.float32))


def test_bias_update_moves_toward_balance():
    # repeated updates on a fixed skewed score profile make the biased
    # selection even out: the bias gap ends opposite to the score gap
    rng = np.random.default_rng(3)
    T, E, k = 256, 8, 2
    base = rng.normal(size=(T, E)).astype(np.float32)
    base[:, 0] += 2.0                       # expert 0 is favoured
    b = np.zeros(E, np.float32)
    loads = []
    for _ in range(200):
        keys = (base + b).astype(np.float32)
        idx = np.stack([O._order_desc(keys[t], list(range(E)))[:k]
                        for t in range(T)])
        cnt = np.bincount(idx.reshape(-1), minlength=E)
        loads.append(cnt.max() - cnt.min())
        b = O.bias_update(b, cnt, T, k, gamma=0.01)
    assert loads[-1] < loads[0] / 4
    assert b[0] < b[1:].min()


# --------------------------------------------------------- dispatch matrix
def test_dispatch_matrix_counts_only_kept_pairs():
    rng = np.random.default_rng(5)
    T, k, E, R, cap = 64, 2, 8, 4, 12
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[:20, 0] = 0                          # force drops on expert 0
    lay = O.dispatch_layout(idx, E, R, cap)
    m = O.dispatch_matrix(idx, 4, R, E, lay["dst_row"])
    assert m.sum() == lay["n_kept"] and lay["dropped"] > 0
    assert (m.sum(axis=0) == lay["rank_send_counts"]).all()
    kept = (lay["dst_row"] >= 0).reshape(T, k)
    assert (m.sum(axis=1) == kept.reshape(4, -1).sum(axis=1)).all()
    m_all = O.dispatch_matrix(idx, 4, R, E)
    assert m_all.sum() == T * k and (m_all >= m).all()


def test_dispatch_matrix_hand_example():
    # the page's worked dispatch example as two source shards of two tokens:
    # idx [[0,2],[1,3],[0,1],[2,3]], E=4, 2 ranks -> rows [[2,2],[2,2]]
    idx = np.array([[0, 2], [1, 3], [0, 1], [2, 3]], np.int32)
    m = O.dispatch_matrix(idx, 2, 2, 4)
    assert m.tolist() == [[2, 2], [2, 2]]
    assert O.dispatch_matrix(idx, 4, 2, 4).tolist() == \
        [[1, 1], [1, 1], [2, 0], [0, 2]]


# ------------------------------------------------------ padded layout -----
@pytest.mark.parametrize("cap", [1, 3, 12])
def test_padded_layout_matches_compact(cap):
    rng = np.random.default_rng(cap)
    T, k, E, D = 20, 2, 5, 6
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = rng.normal(size=(T, D))
    lay = O.dispatch_layout(idx, E, 1, cap)
    pad = O.padded_layout(lay, E, cap)
    xp = O.permute(x, lay["src_pair"], k)
    xpad = O.permute_padded(x, pad["src_pair_padded"], k)
    assert xpad.shape == (E * cap, D)
    for e in range(E):
        c, o = int(lay["counts"][e]), int(lay["offsets"][e])
        np.testing.assert_array_equal(xpad[e * cap:e * cap + c], xp[o:o + c])
        assert (xpad[e * cap + c:(e + 1) * cap] == 0).all()
    # the same combine over either layout gives the same y
    gate = rng.random((T, k))
    y1 = O.combine(xp, lay["dst_row"], gate, T, k)
    y2 = O.combine(xpad, pad["dst_row_padded"], gate, T, k)
    np.testing.assert_array_equal(y1, y2)
    assert ((pad["dst_row_padded"] >= 0) == (lay["dst_row"] >= 0)).all()
    assert (pad["src_pair_padded"] < 0).sum() == E * cap - lay["n_kept"]


def test_padded_ffn_rows_are_zero_for_padding():
    # SwiGLU of a zero row is zero, so the static-shape FFN over the padded
    # buffer equals the compact result on kept rows and 0 elsewhere
    rng = np.random.default_rng(11)
    T, k, E, D, F, cap = 12, 2, 3, 4, 6, 7
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = rng.normal(size=(T, D))
    w13 = rng.normal(size=(E, 2 * F, D))
    w2 = rng.normal(size=(E, D, F))
    lay = O.dispatch_layout(idx, E, 1, cap)
    pad = O.padded_layout(lay, E, cap)
    yp = O.grouped_ffn(O.permute(x, lay["src_pair"], k), lay["offsets"],
                       w13, w2)
    ypad = O.grouped_ffn(O.permute_padded(x, pad["src_pair_padded"], k),
                         pad["offsets_padded"], w13, w2)
    for e in range(E):
        c, o = int(lay["counts"][e]), int(lay["offsets"][e])
        np.testing.assert_allclose(ypad[e * cap:e * cap + c], yp[o:o + c],
                                   rtol=1e-12)
        assert (ypad[e * cap + c:(e + 1) * cap] == 0).all()


# ------------------------------------------------- planted mistakes -------
def _fails(f):
    try:
        f()
    except AssertionError:
        return True
    return False


def test_mutation_f_over_tokens_not_pairs_is_caught(monkeypatch):
    real = O.router_stats

    def wrong(logits, topk_idx, E, mode, alpha):
        st = real(logits, topk_idx, E, mode, alpha)
        k = np.asarray(topk_idx).shape[1]
        st["f"] = st["f"] * k
        st["aux_loss"] = alpha * E * float(np.sum(st["f"] * st["P"]))
        return st
    monkeypatch.setattr(O, "router_stats", wrong)
    assert _fails(lambda: test_aux_loss_is_alpha_at_perfect_balance(
        O.SOFTMAX_TOPK, 16, 2, 8))


def test_mutation_bias_sign_is_caught(monkeypatch):
    real = O.bias_update
    monkeypatch.setattr(O, "bias_update",
                        lambda b, c, T, k, gamma: real(b, c, T, k, -gamma))
    assert _fails(test_bias_update_hand_example)
    assert _fails(test_bias_update_moves_toward_balance)


def test_mutation_padding_not_zeroed_is_caught(monkeypatch):
    real = O.permute_padded

    def ones(x, src, k):
        out = real(x, src, k)
        out[np.asarray(src) < 0] = 1.0
        return out
    monkeypatch.setattr(O, "permute_padded", ones)
    assert _fails(lambda: test_padded_layout_matches_compact(12))


# ------------------------------------------------------ aligned layout -----
@pytest.mark.parametrize("align", [1, 8, 64])
def test_aligned_layout_invariants(align):
    rng = np.random.default_rng(align)
    T, k, E = 300, 2, 7
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[:50, 0] = 3                         # a heavy expert
    lay = O.dispatch_layout(idx, E, 1, 90)
    al = O.aligned_layout(lay, E, align)
    off_a = al["offsets_aligned"]
    assert (off_a % align == 0).all()
    # align = 1 is the compact layout itself
    if align == 1:
        assert off_a.tolist() == lay["offsets"].tolist()
        assert al["dst_row_aligned"].tolist() == lay["dst_row"].tolist()
    dst = al["dst_row_aligned"]
    kept = dst >= 0
    assert (kept == (lay["dst_row"] >= 0)).all()
    assert len(set(dst[kept].tolist())) == kept.sum()      # one row each
    for p in np.flatnonzero(kept):
        e = int(idx.reshape(-1)[p])
        assert off_a[e] <= dst[p] < off_a[e] + lay["counts"][e]
        # same position inside the expert as in the compact layout
        assert dst[p] - off_a[e] == lay["dst_row"][p] - lay["offsets"][e]
    assert off_a[E] <= T * k + (align - 1) * E
