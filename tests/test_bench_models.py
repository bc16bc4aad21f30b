"""CPU checks of the algorithmic work bench.py divides by (the roofline
numerators), against the sizes the source pages' configurations imply:
the Mixtral-like FFN is about 1.44 TFLOP over 2.82 GB of expert weights,
the DeepSeek-like one about 2.89 TFLOP over 22.5 GB, and the T = 65536
permute of the dispatch sweep reads about 0.54 GB and writes about 4.29 GB
("Expert Parallelism in LLMs", The Execution Pipeline, steps 2 and 4; the
configurations' T, D, E, k, F)."""
import importlib.util
import os

import pytest

from combine_router_gemm_top_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"hbm_gbs": 6500.0, "bf16_tflops_sustained": 1350.0}


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location(
        "bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_mixtral_ffn_work(bench):
    wl = W.WORKLOADS["mixtral_bf16"]
    n = wl.T * wl.k                                     # dropless: every pair
    m = bench.kernel_models(wl, n, 2, PEAKS)
    assert m["ffn"]["flops"] == pytest.approx(1.443e12, rel=1e-3)
    weights = wl.E * 3 * wl.F * wl.D * 2
    assert weights == pytest.approx(2.818e9, rel=1e-3)
    assert m["ffn"]["bytes"] == weights + 2 * n * wl.D * 2
    # 1.44 TFLOP against 2.9 GB: above the ridge, so tensor-bound
    assert m["ffn"]["bound"] == "tensor"


def test_deepseek_ffn_work(bench):
    wl = W.WORKLOADS["deepseek_bf16"]
    n = wl.T * wl.k
    m = bench.kernel_models(wl, n, 2, PEAKS)
    assert m["ffn"]["flops"] == pytest.approx(2.886e12, rel=1e-3)
    assert wl.E * 3 * wl.F * wl.D * 2 == pytest.approx(22.55e9, rel=1e-3)
    # 2.9 TFLOP against 23 GB of weights: the weight stream bounds it
    assert m["ffn"]["bound"] == "hbm"


def test_switch_ffn_counts_only_active_experts(bench):
    wl = W.WORKLOADS["switch_bf16"]
    full = bench.kernel_models(wl, 1753, 2, PEAKS)
    part = bench.kernel_models(wl, 1753, 2, PEAKS, active_experts=20)
    per_expert = 3 * wl.F * wl.D * 2
    assert full["ffn"]["bytes"] - part["ffn"]["bytes"] == \
        (wl.E - 20) * per_expert
    assert part["ffn"]["flops"] == full["ffn"]["flops"]


def test_permute_reads_only_tokens_with_a_kept_pair(bench):
    # at capacity a token whose pairs all dropped has no row to move: permute
    # reads t_kept rows, combine still writes all T rows of y (zeros there)
    wl = W.WORKLOADS["switch_bf16"]
    n, t_kept = 1753, 1753                              # k = 1
    m = bench.kernel_models(wl, n, 2, PEAKS, t_kept=t_kept)
    ids = wl.T * wl.k * 4
    assert m["permute"]["bytes"] == (t_kept + n) * wl.D * 2 + ids
    assert m["combine"]["bytes"] == (n + wl.T) * wl.D * 2 + 2 * ids
    dropless = bench.kernel_models(wl, n, 2, PEAKS)
    assert dropless["permute"]["bytes"] == (wl.T + n) * wl.D * 2 + ids


def test_tokens_kept_counts_tokens_with_a_kept_pair(bench):
    # dst_row < 0 marks a dropped pair; a token counts once if any of its k
    # pairs was kept
    import torch

    class FakeLayer:
        T, k = 4, 2
        dst_row = torch.tensor([0, -1, -1, -1, 3, 4, -1, 7, 99, 99],
                               dtype=torch.int32)   # padded past T*k
    assert bench.tokens_kept(FakeLayer()) == 3


def test_sweep_permute_and_combine_bytes(bench):
    wl = W.WORKLOADS["sweep_bf16_uniform_T65536"]
    n = wl.T * wl.k
    m = bench.kernel_models(wl, n, 2, PEAKS)
    assert "ffn" not in m                                # identity experts
    x_bytes = wl.T * wl.D * 2
    xp_bytes = n * wl.D * 2
    assert x_bytes == pytest.approx(0.537e9, rel=1e-3)
    assert xp_bytes == pytest.approx(4.295e9, rel=1e-3)
    ids = wl.T * wl.k * 4
    assert m["permute"]["bytes"] == x_bytes + xp_bytes + ids
    # combine is the mirror: Yp read once, y written once, ids and gates
    assert m["combine"]["bytes"] == xp_bytes + x_bytes + 2 * ids
    for key in ("permute", "combine", "layout"):
        assert m[key]["bound"] == "hbm"


def test_route_work_and_bound(bench):
    wl = W.WORKLOADS["sweep_bf16_uniform_T65536"]
    m = bench.kernel_models(wl, wl.T * wl.k, 2, PEAKS)
    assert m["route"]["flops"] == pytest.approx(68.7e9, rel=1e-3)
    # x (537 MB) dominates the router's bytes; at E = 128 the GEMM stays
    # below the ridge and HBM bounds it
    assert m["route"]["bound"] == "hbm"
    assert m["route"]["roofline_ms"] == pytest.approx(
        m["route"]["bytes"] / (PEAKS["hbm_gbs"] * 1e9) * 1e3)


def test_traffic_keys_match_workload_shapes(bench):
    # each ncu traffic figure is looked up by (workload, T, E, step, FFN
    # variant); a key whose shape or kernel differs from the workload's
    # would never be found
    from combine_router_gemm_top_b300 import _lib as L
    from combine_router_gemm_top_b300 import build as B
    B.build(verbose=False)
    for (name, T, E, step, variant), v in bench.NCU_DRAM_BYTES.items():
        wl = W.WORKLOADS[name]
        assert (wl.T, wl.E) == (T, E), name
        assert step == "ffn" and not wl.identity_experts
        assert L.moe_grouped_ffn_variant(wl.E, wl.D, wl.F, wl.T * wl.k,
                                         L.MOE_BF16) == variant, name
        # a figure of the right order against all experts' weights plus
        # activations: above a quarter of them (the Switch-like layer has 20
        # of 64 experts active) and below 1.5x (the SM-pair kernel's swapped
        # tail tiles re-read their weight tiles: 1.31x measured)
        m = bench.kernel_models(wl, wl.T * wl.k, 2, PEAKS)
        assert 0.25 * m["ffn"]["bytes"] < v < 1.5 * m["ffn"]["bytes"], name


def test_bf16_peak_follows_the_run_regime(bench):
    # the tensor denominator: burst when the timed region is short or the
    # clocks never showed the power cap; sustained for a long capped run
    peaks = {"bf16_tflops": 1775.0, "bf16_tflops_sustained": 1400.0,
             "source": "measured"}
    capped = {"reasons": ["sw_power_cap"]}
    free = {"reasons": []}
    assert bench.choose_bf16_peak(peaks, 0.03, capped)[0] == 1775.0
    assert bench.choose_bf16_peak(peaks, 5.0, free)[0] == 1775.0
    assert bench.choose_bf16_peak(peaks, 5.0, None)[0] == 1775.0
    pk, note = bench.choose_bf16_peak(peaks, 5.0, capped)
    assert pk == 1400.0 and "sustained" in note
    assert "burst" in bench.choose_bf16_peak(peaks, 0.5, capped)[1]


def test_default_run_measures_every_configuration(bench):
    # the default line carries a sub-record for each configuration besides
    # the headline, and every name is a known workload
    names = set(bench.SUB_WORKLOADS)
    assert names == {"deepseek_bf16", "switch_bf16", "tiny_f32",
                     "sweep_bf16_uniform_T65536", "sweep_bf16_zipf_T65536"}
    for n in names:
        assert n in W.WORKLOADS
