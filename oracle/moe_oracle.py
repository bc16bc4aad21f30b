"""CPU oracle for the mixture-of-experts layer forward pass.

TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct numpy in float64.
Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module; the product path never does.  It shares no code,
tables or helpers with the CUDA library.

What it computes (each function cites the passage it follows):

  y_t = sum over the top-k experts i of g_i(x_t) * Expert_i(x_t)
      ("Expert Parallelism in LLMs", section "The Distributed MoE Dilemma:
       Dense vs. Sparse Sharding", the MoE layer equation)

split into the steps of that page's section "The Execution Pipeline":
router gating and top-k (step 1), local permutation into contiguous
per-destination buffers (step 2), the per-expert SwiGLU GEMMs (step 4), and
the un-permute with gated reduction (step 6).  On one device the two
all-to-all-v exchanges (steps 3 and 5) are identities; the oracle emits the
per-rank send counts and displacements the dispatch exchange would take
("All-to-All Communication", the expert_parallel_dispatch listing).

Readings taken where the pages leave a step open (each is also listed in the
design notes):
  * selection key: the fp32 logit in softmax modes (softmax is monotone);
    in sigmoid mode key = fp32(s + b_e), where s = fp32(sigmoid(l)) is the
    sigmoid evaluated in float64 and rounded once to fp32, and the bias is
    added in fp32 (round to nearest even);
  * ties: equal keys go to the lower expert index, equal group scores to the
    lower group index; slot order is descending key;
  * group score: sum of the top `group_score_topk` biased keys of the group,
    added in fp32 in descending-key order;
  * drop priority: pairs are visited in (token, slot) order, pair id
    p = t*k + j; a pair is kept iff fewer than `capacity` earlier pairs chose
    the same expert; gates are not renormalised after a drop;
  * SwiGLU: Expert(h) = W2 (SiLU(W1 h) * (W3 h)) -- the printed form places
    the product inside the SiLU, which would not be a gated unit;
  * the residual is not added (step 6 adds it after the reduction).

Parity pins (see tests/test_oracle_pins.py): the page's worked dispatch
example, brute-force subset enumeration of the selection rule, layout
invariants, identity experts reproducing x, the dense k=E mixture, E=1
against an independent torch SwiGLU, the capacity values printed with the
workloads, and the dispatch/combine element volume 2*T*K*D.
"""
from __future__ import annotations

from fractions import Fraction
import math

import numpy as np

SOFTMAX_TOPK = "softmax_topk"
SOFTMAX_FULL = "softmax_full"
SIGMOID_BIAS = "sigmoid_bias"

F32 = np.float32


# --------------------------------------------------------------------------
# Step 1: router gating ("Expert Parallelism in LLMs", The Execution
# Pipeline, step 1 "Router Gating and Softmax Selection": g_t =
# Softmax(TopK(W_g x_t, k)); "All-to-All Communication", phase 1 "Routing
# decision").
# --------------------------------------------------------------------------
def router_logits(x, w_r, logit_offset=None):
    """logits[t, e] = (W_g x_t)_e, evaluated in float64 from the exact input
    values and rounded once to fp32; an optional per-expert offset is then
    added in fp32 (used to skew the Switch-like workload)."""
    x = np.asarray(x, dtype=np.float64)
    w_r = np.asarray(w_r, dtype=np.float64)
    logits = (x @ w_r.T).astype(F32)
    if logit_offset is not None:
        logits = (logits + np.asarray(logit_offset, dtype=F32)).astype(F32)
    return logits


def sigmoid_f64(logits):
    """sigmoid(l) = 1 / (1 + exp(-l)) in float64 (the definition)."""
    l = np.asarray(logits, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-l))


def sigmoid_f32(logits):
    """fp32(sigmoid(l)): the float64 sigmoid rounded once to fp32.  This is
    the score the sigmoid router ranks by before its bias is added."""
    return sigmoid_f64(logits).astype(F32)


def selection_keys(logits, mode, sel_bias=None):
    """The fp32 value that experts are ranked by.

    softmax modes: the logit (softmax is strictly increasing, so ranking
    logits ranks probabilities without the ties rounding could create).
    sigmoid mode: sigmoid score plus a per-expert bias, the bias steering
    selection only ("Expert Parallelism in LLMs", Modern Dropless Dynamic
    Dispatch: bias terms on routing scores; "Chapter 10: MoE parallelism",
    section 4, aux-loss-free bias adjustment).
    """
    logits = np.asarray(logits, dtype=F32)
    if mode in (SOFTMAX_TOPK, SOFTMAX_FULL):
        return logits.copy()
    if mode == SIGMOID_BIAS:
        s = sigmoid_f32(logits)
        b = np.zeros(logits.shape[-1], F32) if sel_bias is None else \
            np.asarray(sel_bias, dtype=F32)
        return (s + b).astype(F32)
    raise ValueError(mode)


def _order_desc(values, ids):
    """ids sorted by (value descending, id ascending), pure Python."""
    return sorted(ids, key=lambda i: (-float(values[i]), i))


def group_mask(keys_row, n_groups, topk_groups, group_score_topk):
    """Group-limited routing: experts form n_groups contiguous groups; each
    group is scored by the fp32 sum of its `group_score_topk` largest keys
    (largest first); the `topk_groups` best groups stay eligible.  This is
    the limit on how many destinations a token may reach, chosen before the
    per-expert selection ("Expert Parallelism and All-to-All", Three ways the
    system fights back: a token may reach at most 4 nodes, chosen before the
    per-expert selection).  Returns a boolean eligibility mask over experts.
    """
    E = len(keys_row)
    if n_groups <= 1:
        return np.ones(E, dtype=bool)
    gsize = E // n_groups
    scores = []
    for g in range(n_groups):
        members = list(range(g * gsize, (g + 1) * gsize))
        top = _order_desc(keys_row, members)[:group_score_topk]
        acc = F32(0.0)
        for i in top:
            acc = F32(acc + keys_row[i])
        scores.append(acc)
    chosen = _order_desc(scores, list(range(n_groups)))[:topk_groups]
    mask = np.zeros(E, dtype=bool)
    for g in chosen:
        mask[g * gsize:(g + 1) * gsize] = True
    return mask


def route_from_logits(logits, k, mode, sel_bias=None, n_groups=1,
                      topk_groups=1, group_score_topk=0):
    """Top-k selection and gates for every token from fp32 logits [T, E].

    Returns (topk_idx int32 [T, k], topk_gate float64 [T, k]).
      softmax_topk : g = softmax over the k selected logits
                     (g_t = Softmax(TopK(W_g x_t, k)))
      softmax_full : g = p_e, softmax over all E experts (k=1 Switch gate)
      sigmoid_bias : g_j = s_j / sum of the selected s, with the unbiased
                     sigmoid score s
    """
    logits = np.asarray(logits, dtype=F32)
    T, E = logits.shape
    keys = selection_keys(logits, mode, sel_bias)
    idx = np.zeros((T, k), dtype=np.int32)
    gate = np.zeros((T, k), dtype=np.float64)
    l64 = logits.astype(np.float64)
    for t in range(T):
        mask = group_mask(keys[t], n_groups, topk_groups, group_score_topk)
        eligible = [e for e in range(E) if mask[e]]
        sel = _order_desc(keys[t], eligible)[:k]
        idx[t] = sel
        if mode == SOFTMAX_TOPK:
            z = l64[t, sel]
            w = np.exp(z - z.max())
            gate[t] = w / w.sum()
        elif mode == SOFTMAX_FULL:
            w = np.exp(l64[t] - l64[t].max())
            p = w / w.sum()
            gate[t] = p[sel]
        else:
            s = sigmoid_f64(l64[t, sel])
            gate[t] = s / s.sum()
    return idx, gate


# --------------------------------------------------------------------------
# Capacity ("Expert Parallelism in LLMs", Static Capacity Factors and Token
# Dropping: C_expert = ceil(CF * k * B * S / E)).
# --------------------------------------------------------------------------
def expert_capacity(capacity_factor, T, k, E):
    """ceil(CF * k * T / E) in exact rational arithmetic; None -> dropless."""
    if capacity_factor is None:
        return None
    cf = Fraction(str(capacity_factor))
    return math.ceil(cf * k * T / E)


# --------------------------------------------------------------------------
# Step 2: local permutation layout ("Expert Parallelism in LLMs", The
# Execution Pipeline, step 2 "Local Token Permutation"; "All-to-All
# Communication", expert_parallel_dispatch listing: destination device =
# expert // experts_per_device, sorted by destination, bincount of
# destinations as the send counts).
# --------------------------------------------------------------------------
def dispatch_layout(topk_idx, E, R, capacity=None):
    """Binning of the T*k (token, expert) pairs into an expert-contiguous
    buffer, walking pairs in (token, slot) order.

    Returns a dict:
      counts      [E]   kept pairs per expert
      counts_raw  [E]   routed pairs per expert before the capacity clamp
      offsets     [E+1] exclusive scan of counts (start row of each expert)
      dst_row     [P]   buffer row of pair p, or -1 if the pair was dropped
      src_pair    [N]   pair id stored in each buffer row
      n_kept, dropped
      rank_send_counts [R], rank_send_displs [R]: rows bound for each
                  virtual expert-parallel rank (experts in contiguous blocks
                  of E/R), the send split of the dispatch all-to-all-v
    """
    idx = np.asarray(topk_idx).reshape(-1)
    P = idx.shape[0]
    cap = None if (capacity is None or capacity <= 0) else int(capacity)
    seen = [0] * E
    pos = [0] * P
    keep = [False] * P
    for p in range(P):
        e = int(idx[p])
        pos[p] = seen[e]
        keep[p] = cap is None or seen[e] < cap
        seen[e] += 1
    counts_raw = np.array(seen, dtype=np.int64)
    counts = counts_raw.copy() if cap is None else np.minimum(counts_raw, cap)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    n_kept = int(offsets[E])
    dst_row = np.full(P, -1, dtype=np.int64)
    src_pair = np.full(n_kept, -1, dtype=np.int64)
    for p in range(P):
        if keep[p]:
            r = int(offsets[int(idx[p])]) + pos[p]
            dst_row[p] = r
            src_pair[r] = p
    epr = E // R
    rank_counts = np.array([int(counts[r * epr:(r + 1) * epr].sum())
                            for r in range(R)], dtype=np.int64)
    rank_displs = np.zeros(R, dtype=np.int64)
    for r in range(1, R):
        rank_displs[r] = rank_displs[r - 1] + rank_counts[r - 1]
    return dict(counts=counts, counts_raw=counts_raw, offsets=offsets,
                dst_row=dst_row, src_pair=src_pair, n_kept=n_kept,
                dropped=P - n_kept, rank_send_counts=rank_counts,
                rank_send_displs=rank_displs)


def dispatch_matrix(topk_idx, n_src, n_dst, E, dst_row=None):
    """Pairs sent from each source shard to each destination rank: tokens
    are split into n_src equal contiguous shards, experts into n_dst
    contiguous blocks ("All-to-All Communication", the routing simulation
    listing and its printed dispatch matrix).  With dst_row given, only
    kept pairs (dst_row >= 0) are counted: a dropped pair is never sent."""
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    per_src = T // n_src
    epr = E // n_dst
    m = np.zeros((n_src, n_dst), dtype=np.int64)
    for t in range(T):
        s = t // per_src
        for j in range(k):
            if dst_row is not None and int(dst_row[t * k + j]) < 0:
                continue
            m[s, int(idx[t, j]) // epr] += 1
    return m


def permute(x, src_pair, k):
    """xp[r] = x[src_pair[r] // k]: each buffer row is a copy of its token."""
    x = np.asarray(x, dtype=np.float64)
    return np.stack([x[int(p) // k] for p in src_pair]) if len(src_pair) \
        else np.zeros((0, x.shape[1]))


# --------------------------------------------------------------------------
# Step 4: local expert computation ("Expert Parallelism in LLMs", The
# Execution Pipeline, step 4 "Local Expert Computation": tokens of one expert
# packed into one batched GEMM; h_out = W2 . SiLU(W1 h) * (W3 h) under the
# SwiGLU reading above).
# --------------------------------------------------------------------------
def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_expert(h, w1, w3, w2):
    """Rows of h [n, D] through one expert: W1, W3 [F, D], W2 [D, F]."""
    h = np.asarray(h, dtype=np.float64)
    gate = h @ np.asarray(w1, dtype=np.float64).T
    up = h @ np.asarray(w3, dtype=np.float64).T
    return (silu(gate) * up) @ np.asarray(w2, dtype=np.float64).T


def split_w13(w13_e):
    """w13 rows 0..F-1 are W1 (gate), rows F..2F-1 are W3 (up)."""
    F = w13_e.shape[0] // 2
    return w13_e[:F], w13_e[F:]


def grouped_ffn(xp, offsets, w13, w2):
    """Apply expert e to its contiguous rows [offsets[e], offsets[e+1])."""
    xp = np.asarray(xp, dtype=np.float64)
    yp = np.zeros_like(xp)
    E = len(offsets) - 1
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            w1, w3 = split_w13(w13[e])
            yp[a:b] = swiglu_expert(xp[a:b], w1, w3, w2[e])
    return yp


# --------------------------------------------------------------------------
# Step 6: un-permutation and weighted reduction ("Expert Parallelism in
# LLMs", The Execution Pipeline, step 6: restore positions, multiply by the
# gate, sum the k outputs; the residual is added afterwards, outside).
# --------------------------------------------------------------------------
def combine(yp, dst_row, gate, T, k):
    """y[t] = sum over kept slots j of gate[t, j] * yp[dst_row[t*k + j]];
    dropped pairs (dst_row = -1) contribute nothing ("Static Capacity
    Factors and Token Dropping": dropped tokens bypass the expert layer)."""
    yp = np.asarray(yp, dtype=np.float64)
    D = yp.shape[1]
    y = np.zeros((T, D), dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = int(dst_row[t * k + j])
            if r >= 0:
                y[t] += gate[t, j] * yp[r]
    return y


def moe_forward(x, w_r, k, E, R, mode, w13=None, w2=None, sel_bias=None,
                logit_offset=None, n_groups=1, topk_groups=1,
                group_score_topk=0, capacity=None, logits=None,
                topk_idx=None, topk_gate=None):
    """The whole layer.  With logits given, routing starts from those fp32
    values; with topk_idx/topk_gate given, routing is skipped (pre-drawn
    routing).  w13 = None means identity experts (Expert_i(h) = h)."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    out = {}
    if topk_idx is None:
        if logits is None:
            logits = router_logits(x, w_r, logit_offset)
        topk_idx, topk_gate = route_from_logits(
            logits, k, mode, sel_bias, n_groups, topk_groups,
            group_score_topk)
        out["logits"] = logits
    out["topk_idx"] = np.asarray(topk_idx, dtype=np.int32)
    out["topk_gate"] = np.asarray(topk_gate, dtype=np.float64)
    lay = dispatch_layout(topk_idx, E, R, capacity)
    out.update(lay)
    xp = permute(x, lay["src_pair"], k)
    out["xp"] = xp
    yp = xp if w13 is None else grouped_ffn(xp, lay["offsets"], w13, w2)
    out["yp"] = yp
    out["y"] = combine(yp, lay["dst_row"], topk_gate, T, k)
    return out


def token_output(x_t, t, topk_idx, topk_gate, dst_row, k, expert_weights):
    """y for a single token straight from the layer equation, with
    expert_weights(e) -> (w1, w3, w2) in float64 (or None for identity
    experts).  Used to check sampled tokens of large workloads."""
    x_t = np.asarray(x_t, dtype=np.float64)[None, :]
    y = np.zeros(x_t.shape[1])
    for j in range(k):
        if int(dst_row[t * k + j]) < 0:
            continue
        e = int(topk_idx[t][j])
        ws = expert_weights(e)
        h = x_t if ws is None else swiglu_expert(x_t, *ws)
        y += float(topk_gate[t][j]) * h[0]
    return y


def dispatch_combine_volume(T, k, D):
    """V_layer = 2 * B * S * K * D elements ("Communication Overhead
    Analysis", the V_layer equation): every pair goes out once and comes
    back once."""
    return 2 * T * k * D


def dispatch_bytes_per_rank(T, k, D, ep, elem_bytes):
    """Per-device dispatch volume B*S*k*H*(EP-1)/EP*sizeof ("Expert
    Parallelism in LLMs", Communication Volume and Hardware Topology), for
    uniform routing."""
    return Fraction(T * k * D * (ep - 1) * elem_bytes, ep)


# --------------------------------------------------------------------------
# Router statistics ("Expert Parallelism in LLMs", Static Capacity Factors
# and Token Dropping: the auxiliary load-balancing loss
# L_aux = alpha * E * sum_i f_i * P_i; Modern Dropless Dynamic Dispatch:
# dynamically adjusted bias terms on the routing scores).
# --------------------------------------------------------------------------
def router_probabilities(logits, mode):
    """The router probability each token gives every expert, float64 [T, E].

    softmax modes: p = softmax of the token's E logits.
    sigmoid mode: p = s / sum over all E of s, with s = sigmoid(logit), the
    scores normalised to a distribution over experts (reading: the pages
    define P_i only as "the router probability allocated to expert i")."""
    l64 = np.asarray(logits, dtype=np.float64)
    out = np.zeros_like(l64)
    for t in range(l64.shape[0]):
        if mode == SIGMOID_BIAS:
            s = sigmoid_f64(l64[t])
            out[t] = s / s.sum()
        else:
            w = np.exp(l64[t] - l64[t].max())
            out[t] = w / w.sum()
    return out


def router_stats(logits, topk_idx, E, mode, alpha):
    """f_i, P_i and L_aux of one routing decision.

      counts_routed[i] = pairs that selected expert i (before any capacity
                         drop: "fraction of tokens dispatched" is read as
                         the routing decision itself)
      f_i = counts_routed[i] / (T * k)     (sums to 1)
      P_i = mean over tokens of the router probability of expert i
      L_aux = alpha * E * sum_i f_i * P_i
    With perfectly even routing and even probabilities L_aux = alpha."""
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[int(idx[t, j])] += 1
    f = counts / float(T * k) if T * k else np.zeros(E)
    p = router_probabilities(logits, mode)
    P = p.mean(axis=0) if T else np.zeros(E)
    loss = alpha * E * float(np.sum(f * P))
    return dict(counts_routed=counts, f=f, P=P, aux_loss=loss)


def bias_update(bias, counts_routed, T, k, gamma):
    """Auxiliary-loss-free balancing step on the selection bias: an expert
    whose routed load is above the mean load T*k/E has its bias lowered by
    gamma, one below it raised by gamma, one exactly at it left alone
    (reading: the pages say only that the bias terms are adjusted
    dynamically to keep the load balanced; this is the plainest rule that
    moves every expert toward the mean).  The comparison is exact integer
    arithmetic: sign(T*k - E*load)."""
    b = np.asarray(bias, dtype=F32).copy()
    E = b.shape[0]
    for e in range(E):
        d = T * k - E * int(counts_routed[e])
        if d > 0:
            b[e] = F32(b[e] + F32(gamma))
        elif d < 0:
            b[e] = F32(b[e] - F32(gamma))
    return b


# --------------------------------------------------------------------------
# Static-capacity padded layout ("Expert Parallelism in LLMs", Static
# Capacity Factors and Token Dropping: fixed per-expert buffers of
# C_expert rows; unused slots are padding).
# --------------------------------------------------------------------------
def padded_layout(layout, E, capacity):
    """Row of each kept pair in a [E, C, D] buffer: expert e owns rows
    [e*C, (e+1)*C) and its kept pairs fill them in the compact layout's
    order.  Returns dst_row_padded [P] (-1 if dropped), src_pair_padded
    [E*C] (-1 for a padding row) and the uniform offsets e*C."""
    cap = int(capacity)
    dst = np.asarray(layout["dst_row"])
    off = np.asarray(layout["offsets"])
    src = np.asarray(layout["src_pair"])
    counts = np.asarray(layout["counts"])
    dst_p = np.full(dst.shape[0], -1, dtype=np.int64)
    src_p = np.full(E * cap, -1, dtype=np.int64)
    for e in range(E):
        for pos in range(int(counts[e])):
            p = int(src[int(off[e]) + pos])
            dst_p[p] = e * cap + pos
            src_p[e * cap + pos] = p
    return dict(dst_row_padded=dst_p, src_pair_padded=src_p,
                offsets_padded=np.arange(E + 1, dtype=np.int64) * cap)


def permute_padded(x, src_pair_padded, k):
    """xpad[r] = x[src_pair_padded[r] // k], zeros for padding rows."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros((len(src_pair_padded), x.shape[1]))
    for r, p in enumerate(src_pair_padded):
        if int(p) >= 0:
            out[r] = x[int(p) // k]
    return out


# --------------------------------------------------------------------------
# Backward pass ("Expert Parallelism in LLMs", Backward Pass Symmetry: the
# upstream gradient dL/dy goes to the experts along the dispatch pattern,
# the experts form their weight gradients and input gradients, and the
# input gradients return along the combine pattern).  The routing decision
# (which experts, which pairs are kept) is piecewise constant in x, so the
# gradient flows through the gates and the experts with the selection
# fixed; that is the plain chain rule of the layer equation
#     y_t = sum over kept slots j of g_j(x_t) * Expert_{e_j}(x_t).
# --------------------------------------------------------------------------
def silu_grad(z):
    """d/dz [z * sigmoid(z)] = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def expert_backward(h, w1, w3, w2, dout):
    """Gradients of out = W2 (SiLU(W1 h) * (W3 h)) for rows h [n, D] given
    dout [n, D]: returns dh [n, D], dw1, dw3 [F, D], dw2 [D, F]."""
    h = np.asarray(h, dtype=np.float64)
    w1, w3, w2 = (np.asarray(w, dtype=np.float64) for w in (w1, w3, w2))
    dout = np.asarray(dout, dtype=np.float64)
    g = h @ w1.T
    u = h @ w3.T
    act = silu(g) * u
    dact = dout @ w2                      # [n, F]
    dw2 = dout.T @ act                    # [D, F]
    du = dact * silu(g)
    dg = dact * u * silu_grad(g)
    dh = dg @ w1 + du @ w3
    dw1 = dg.T @ h
    dw3 = du.T @ h
    return dh, dw1, dw3, dw2


def gate_backward(logits_row, sel, dgate, mode):
    """dL/dlogits of one token from dL/dgate of its k selected slots.

      softmax_topk: g = softmax over the selected logits
      softmax_full: g_j = p_{e_j}, p = softmax over all E logits
      sigmoid_bias: g_j = s_j / sum_sel s, s = sigmoid(logit) (the bias
                    only selects, so it has no gradient path)
    """
    l = np.asarray(logits_row, dtype=np.float64)
    dgate = np.asarray(dgate, dtype=np.float64)
    dl = np.zeros_like(l)
    sel = [int(e) for e in sel]
    if mode == SOFTMAX_TOPK:
        z = l[sel]
        w = np.exp(z - z.max())
        g = w / w.sum()
        dl[sel] = g * (dgate - float(g @ dgate))
    elif mode == SOFTMAX_FULL:
        w = np.exp(l - l.max())
        p = w / w.sum()
        dp = np.zeros_like(l)
        for j, e in enumerate(sel):
            dp[e] += dgate[j]
        dl = p * (dp - float(p @ dp))
    else:
        s = sigmoid_f64(l[sel])
        S = s.sum()
        g = s / S
        ds = (dgate - float(g @ dgate)) / S
        dl[sel] = ds * s * (1.0 - s)
    return dl


def moe_backward(x, w_r, dy, k, E, R, mode, w13=None, w2=None,
                 sel_bias=None, logit_offset=None, n_groups=1,
                 topk_groups=1, group_score_topk=0, capacity=None,
                 logits=None):
    """Gradients of L = sum(dy * y) for the layer of moe_forward.

    Returns dx [T, D], dw_r [E, D], dw13 [E, 2F, D], dw2 [E, D, F] (None for
    identity experts), and the intermediates dgate [T, k] (0 for dropped
    pairs), dlogits [T, E], dyp [N, D] (the gate-scaled upstream gradient in
    the expert-contiguous order) and dxp [N, D] (the experts' input
    gradients in that order)."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, D = x.shape
    fw = moe_forward(x, w_r, k, E, R, mode, w13=w13, w2=w2,
                     sel_bias=sel_bias, logit_offset=logit_offset,
                     n_groups=n_groups, topk_groups=topk_groups,
                     group_score_topk=group_score_topk, capacity=capacity,
                     logits=logits)
    idx, gate = fw["topk_idx"], fw["topk_gate"]
    dst, off, src = fw["dst_row"], fw["offsets"], fw["src_pair"]
    xp, yp = fw["xp"], fw["yp"]
    N = len(src)
    # dispatch of the upstream gradient: dyp[r] = g * dy[t]; dgate = dy . yp
    dyp = np.zeros((N, D))
    dgate = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            r = int(dst[t * k + j])
            if r >= 0:
                dyp[r] = gate[t, j] * dy[t]
                dgate[t, j] = float(dy[t] @ yp[r])
    # experts
    dxp = dyp.copy() if w13 is None else np.zeros((N, D))
    dw13 = dw2 = None
    if w13 is not None:
        F = np.asarray(w13[0]).shape[0] // 2
        dw13 = np.zeros((E, 2 * F, D))
        dw2 = np.zeros((E, D, F))
        for e in range(E):
            a, b = int(off[e]), int(off[e + 1])
            if b > a:
                w1, w3 = split_w13(np.asarray(w13[e], dtype=np.float64))
                dh, dw1, dw3, dw2e = expert_backward(xp[a:b], w1, w3, w2[e],
                                                     dyp[a:b])
                dxp[a:b] = dh
                dw13[e, :F] = dw1
                dw13[e, F:] = dw3
                dw2[e] = dw2e
    # combine of the input gradients: dx[t] = sum over kept j of dxp[row]
    dx = np.zeros((T, D))
    for t in range(T):
        for j in range(k):
            r = int(dst[t * k + j])
            if r >= 0:
                dx[t] += dxp[r]
    # router
    lg = fw["logits"] if "logits" in fw else logits
    dlogits = np.zeros((T, E))
    for t in range(T):
        dlogits[t] = gate_backward(lg[t], idx[t], dgate[t], mode)
    dw_r = dlogits.T @ x
    dx += dlogits @ np.asarray(w_r, dtype=np.float64)
    return dict(dx=dx, dw_r=dw_r, dw13=dw13, dw2=dw2, dgate=dgate,
                dlogits=dlogits, dyp=dyp, dxp=dxp, forward=fw)


def aligned_layout(layout, E, align):
    """The training layout: expert e's rows start at the exclusive scan of
    its kept count rounded up to `align`, in the compact layout's order, so
    that no block of `align` rows holds two experts.  Returns
    dst_row_aligned [P] (-1 if dropped) and offsets_aligned [E+1]."""
    counts = np.asarray(layout["counts"])
    off = np.asarray(layout["offsets"])
    dst = np.asarray(layout["dst_row"])
    idx_of_row = {}
    for e in range(E):
        for r in range(int(off[e]), int(off[e + 1])):
            idx_of_row[r] = e
    off_a = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        c = int(counts[e])
        off_a[e + 1] = off_a[e] + (c + align - 1) // align * align
    dst_a = np.full(dst.shape[0], -1, dtype=np.int64)
    for p, r in enumerate(dst):
        if int(r) >= 0:
            e = idx_of_row[int(r)]
            dst_a[p] = off_a[e] + (int(r) - int(off[e]))
    return dict(dst_row_aligned=dst_a, offsets_aligned=off_a)
