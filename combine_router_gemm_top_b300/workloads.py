"""Seeded synthetic inputs for the MoE-layer forward pass.

This module only draws random numbers and names workload shapes.  It holds
none of the layer's arithmetic (no routing, no layout, no expert math), so the
CUDA path and the CPU oracle can both be fed from it without sharing any of
the method.

Workloads (shapes follow the pages' model families: Mixtral-like top-2,
DeepSeek-V3-like fine-grained top-8, Switch-like top-1 with a capacity factor;
"Expert Parallelism in LLMs", section "Managing Token Imbalance"):

  tiny_f32        T=256   D=64   E=8   k=2 F=128   fp32, softmax top-2, CF 1.25, R=4
  mixtral_bf16    T=2048  D=4096 E=8   k=2 F=14336 bf16, softmax top-2, dropless, R=8
  deepseek_bf16   T=4096  D=7168 E=256 k=8 F=2048  bf16, sigmoid+bias, 8 groups/top-4, R=8
  switch_bf16     T=16384 D=1024 E=64  k=1 F=4096  bf16, full softmax, CF 1.0, skewed, R=16
  sweep_bf16      T in {4096,16384,65536} D=4096 E=128 k=8, identity experts,
                  uniform or Zipf(1.2) expert draws, Dirichlet(1) gates, R=8

Random draws use torch.Generator objects seeded per tensor in a fixed order
(x, w_r, bias, w13, w2, routing), so a (workload, seed, device) triple always
yields the same tensors.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SCORE_SOFTMAX_TOPK = "softmax_topk"
SCORE_SOFTMAX_FULL = "softmax_full"
SCORE_SIGMOID_BIAS = "sigmoid_bias"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    E: int
    k: int
    F: int
    dtype: str                      # "f32" or "bf16"
    score: str                      # one of the SCORE_* names
    R: int                          # virtual expert-parallel ranks
    capacity_factor: Optional[float] = None   # None: dropless
    n_groups: int = 1
    topk_groups: int = 1
    group_score_topk: int = 0
    x_std: float = 1.0
    w_r_std: Optional[float] = None           # None: 1/sqrt(D)
    w_std: Optional[float] = None             # None: 1/sqrt(D)
    bias_range: Optional[float] = None        # selection bias U(-a, a)
    skew: Optional[float] = None              # logit offset skew*log(1/(e+1))
    identity_experts: bool = False
    routing: Optional[str] = None             # "uniform" / "zipf" for sweep
    zipf_s: float = 1.2
    seed: int = 0

    @property
    def P(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _wl_tiny():
    return Workload("tiny_f32", T=256, D=64, E=8, k=2, F=128, dtype="f32",
                    score=SCORE_SOFTMAX_TOPK, R=4, capacity_factor=1.25,
                    w_r_std=0.02, w_std=0.02, seed=0)


def _wl_mixtral():
    return Workload("mixtral_bf16", T=2048, D=4096, E=8, k=2, F=14336,
                    dtype="bf16", score=SCORE_SOFTMAX_TOPK, R=8, seed=1)


def _wl_deepseek():
    return Workload("deepseek_bf16", T=4096, D=7168, E=256, k=8, F=2048,
                    dtype="bf16", score=SCORE_SIGMOID_BIAS, R=8,
                    n_groups=8, topk_groups=4, group_score_topk=2,
                    bias_range=0.1, seed=2)


def _wl_switch():
    return Workload("switch_bf16", T=16384, D=1024, E=64, k=1, F=4096,
                    dtype="bf16", score=SCORE_SOFTMAX_FULL, R=16,
                    capacity_factor=1.0, skew=1.5, seed=3)


def _wl_sweep(T: int, routing: str):
    return Workload(f"sweep_bf16_{routing}_T{T}", T=T, D=4096, E=128, k=8,
                    F=0, dtype="bf16", score=SCORE_SOFTMAX_TOPK, R=8,
                    identity_experts=True, routing=routing, seed=4)


WORKLOADS = {
    "tiny_f32": _wl_tiny(),
    "mixtral_bf16": _wl_mixtral(),
    "deepseek_bf16": _wl_deepseek(),
    "switch_bf16": _wl_switch(),
}
for _T in (4096, 16384, 65536):
    for _r in ("uniform", "zipf"):
        _w = _wl_sweep(_T, _r)
        WORKLOADS[_w.name] = _w


def torch_dtype(wl: Workload) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream * 7_919)
    return g


def _normal(shape, std, gen, device, dtype, chunk=1 << 26):
    """N(0, std^2) samples drawn in fp32 then cast, in row chunks to bound
    temporary memory for multi-GB weight tensors."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=gen, device=device,
                          dtype=torch.float32)
        tmp.mul_(std)
        flat[s:e].copy_(tmp)
    return out


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None,
                with_experts: bool = True) -> dict:
    """Draws every input of one layer pass for workload ``wl``.

    Returns a dict with
      x        [T, D]        activations (fp32 or bf16)
      w_r      [E, D]        router weight, K-major (same dtype as x)
      sel_bias [E] fp32      selection-only bias (sigmoid mode) or None
      logit_offset [E] fp32  per-expert logit offset (skewed mode) or None
      w13      [E, 2F, D]    rows 0..F-1 gate (W1), rows F..2F-1 up (W3)
      w2       [E, D, F]     down projection, K-major
      topk_idx / topk_gate   pre-drawn routing (sweep workloads only)
    """
    seed = wl.seed if seed is None else seed
    dt = torch_dtype(wl)
    T, D, E, F = wl.T, wl.D, wl.E, wl.F
    out = {}
    out["x"] = _normal((T, D), wl.x_std, _gen(seed, 0, device), device, dt)
    wr_std = wl.w_r_std if wl.w_r_std is not None else 1.0 / math.sqrt(D)
    out["w_r"] = _normal((E, D), wr_std, _gen(seed, 1, device), device, dt)
    if wl.bias_range is not None:
        g = _gen(seed, 2, device)
        b = torch.rand(E, generator=g, device=device, dtype=torch.float32)
        out["sel_bias"] = (b * 2.0 - 1.0) * wl.bias_range
    else:
        out["sel_bias"] = None
    if wl.skew is not None:
        ranks = torch.arange(1, E + 1, dtype=torch.float64)
        out["logit_offset"] = (wl.skew * torch.log(1.0 / ranks)).to(
            torch.float32).to(device)
    else:
        out["logit_offset"] = None
    if with_experts and not wl.identity_experts:
        w_std = wl.w_std if wl.w_std is not None else 1.0 / math.sqrt(D)
        out["w13"] = _normal((E, 2 * F, D), w_std, _gen(seed, 3, device),
                             device, dt)
        out["w2"] = _normal((E, D, F), w_std, _gen(seed, 4, device),
                            device, dt)
    else:
        out["w13"] = None
        out["w2"] = None
    if wl.routing is not None:
        idx, gate = draw_routing(T, E, wl.k, wl.routing, wl.zipf_s,
                                 _gen(seed, 5, device), device)
        out["topk_idx"] = idx
        out["topk_gate"] = gate
    return out


def draw_routing(T, E, k, kind, zipf_s, gen, device):
    """k distinct experts per token, uniform or Zipf(s) over expert rank e+1
    (Gumbel-top-k sampling without replacement), slots in draw order, and
    gates drawn from Dirichlet(1) over the k slots (normalised Exp(1))."""
    if kind == "uniform":
        logw = torch.zeros(E, dtype=torch.float64)
    elif kind == "zipf":
        r = torch.arange(1, E + 1, dtype=torch.float64)
        logw = -zipf_s * torch.log(r)
    else:
        raise ValueError(kind)
    u = torch.rand((T, E), generator=gen, device=device, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    keys = gumbel + logw.to(device)
    idx = torch.topk(keys, k, dim=1).indices.to(torch.int32)
    ex = torch.rand((T, k), generator=gen, device=device, dtype=torch.float64)
    ex = -torch.log(ex.clamp_min(1e-300))
    gate = (ex / ex.sum(dim=1, keepdim=True)).to(torch.float32)
    return idx.contiguous(), gate.contiguous()
