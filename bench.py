"""Benchmark of the MoE-layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--only]

A step is one whole layer pass (route -> dispatch layout -> permute ->
grouped SwiGLU FFN -> combine) over one batch of seeded synthetic input with
every input resident in HBM.  The headline workload is the Mixtral-like
top-2 layer (T=2048, D=4096, E=8, k=2, F=14336, bf16, dropless).  After an
eager warm-up, one step is captured as a CUDA graph: a 256 MiB write (> the
126 MB L2, so every step starts with a cold L2), then the five calls with
timing events recorded inside the graph between them.  The timed loop
replays such graphs back to back; the stage times are device time with no
launch boundary between stages, and the flush lies outside them.  The
end-to-end figure ("e2e") is taken through the public layer API with host
copies.

The default run also measures the other configurations the same way (the
DeepSeek-like and Switch-like layers, the tiny fp32 layer, and the T=65536
dispatch/combine sweep with uniform and Zipf routing) and reports each as a
sub-record under "workloads"; --only measures --workload alone.  Tensor-bound
kernels are reported against the measured bf16 burst peak when the timed
region is short or never reached the power cap, else against the sustained
one ("peak_note" says which).

Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs an
independent replica on its own GPU with its own seed (weak scaling, no
collective on the data path); the time is the max over ranks.

--impl reference times the CPU oracle (the reference arm of this
comparison) on the host cores on a bounded token sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at 1 B300; permute+combine GB/s as % of HBM peak"
FLUSH_BYTES = 256 << 20
# A bounded GPU spin (about 0.5 ms) before each isolated call of the extras:
# while it runs the host enqueues the call, so its events measure device time
# and not the Python launch path.  It sits outside the timed events.
HOST_AHEAD_CYCLES = 1_000_000


def host_ahead():
    import torch
    torch.cuda._sleep(HOST_AHEAD_CYCLES)


GRAPH_RING = 4   # step graphs in flight (see run_step_graphs)


def capture_step_graphs(stages, flush, dev, ring=GRAPH_RING):
    """Captures `ring` copies of one step as CUDA graphs: the L2 flush, then
    every stage (a function of the stream) between timing events recorded
    inside the graph (external event-record nodes), so the stage times are
    device time with no launch boundary between stages.  The stages
    allocate nothing and never synchronise, and the eager warm-up before
    this has set every kernel's shared-memory limit.  Returns a list of
    (graph, events)."""
    import torch
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    out = []
    for _ in range(ring):
        evs = [torch.cuda.Event(enable_timing=True, external=True)
               for _ in range(len(stages) + 1)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            flush.zero_()
            for j, fn in enumerate(stages):
                evs[j].record(s)
                fn(s)
            evs[-1].record(s)
        out.append((g, evs))
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return out


def run_step_graphs(graphs, K):
    """Replays the step graphs round-robin K times on the current stream and
    returns the stage times of every step, [K][stages] in ms.  Before a
    graph is replayed again the host reads the times its previous replay
    recorded, so the GPU queue stays len(graphs) - 1 steps deep and the GPU
    never waits for the host."""
    import torch
    R = len(graphs)
    times = []

    def collect(evs):
        times.append([evs[j].elapsed_time(evs[j + 1])
                      for j in range(len(evs) - 1)])

    for i in range(K):
        g, evs = graphs[i % R]
        if i >= R:
            evs[-1].synchronize()
            collect(evs)
        g.replay()
    torch.cuda.synchronize()
    for i in range(max(0, K - R), K):
        collect(graphs[i % R][1])
    return times


def choose_bf16_peak(peaks, wall_s, clk):
    """The dense bf16 denominator for this run's regime: the burst figure
    when the timed region is short (under 1 s) or the sampled clocks never
    showed sw_power_cap, the sustained (power-capped) figure otherwise."""
    capped = clk is not None and "sw_power_cap" in clk.get("reasons", [])
    if wall_s < 1.0 or not capped:
        why = (f"timed region {wall_s:.2f} s" if wall_s < 1.0 else
               "no sw_power_cap in the sampled clocks")
        return peaks["bf16_tflops"], f"bf16 burst ({why}), {peaks['source']}"
    return peaks["bf16_tflops_sustained"], (
        f"bf16 sustained (timed region {wall_s:.2f} s at sw_power_cap), "
        f"{peaks['source']}")


K_graph_cap = 200

# dram__bytes_read.sum + dram__bytes_write.sum per launch from ncu, keyed by
# (workload, T, E, step, FFN variant as moe_grouped_ffn_variant reports it),
# for the grouped FFN's one launch (up and down projection):
#   Mixtral-like   3.5955 GB read + 187.4 MB written (SM pairs)
#   DeepSeek-like 23.3931 GB read + 598.7 MB written (one SM per tile)
#   Switch-like    522.6 MB read +  17.4 MB written (one SM per tile)
NCU_DRAM_BYTES = {("mixtral_bf16", 2048, 8, "ffn", 3): 3.3364e9,
                  ("deepseek_bf16", 4096, 256, "ffn", 2): 2.39966e10,
                  ("switch_bf16", 16384, 64, "ffn", 2): 5.3954e8}

# tokens of the bounded CPU-oracle sample, per workload (about 10-30 s of
# host work)
CPU_SAMPLE_TOKENS = {"tiny_f32": 256, "mixtral_bf16": 48,
                     "deepseek_bf16": 16, "switch_bf16": 512}
# smaller per-step samples for the --impl reference arm, which runs K steps
REF_SAMPLE_TOKENS = {"tiny_f32": 256, "mixtral_bf16": 8,
                     "deepseek_bf16": 4, "switch_bf16": 128}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]),
                    bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p["bf16_tflops_sustained"]),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6400.0, bf16_tflops=1800.0,
                    bf16_tflops_sustained=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def build_layer(wl, device, seed):
    import torch
    from combine_router_gemm_top_b300 import workloads as W
    from combine_router_gemm_top_b300.layer import MoELayer
    inp = W.make_inputs(wl, device=device, seed=seed)
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"], inp["w13"],
                     inp["w2"], F=wl.F, score=wl.score,
                     sel_bias=inp["sel_bias"],
                     logit_offset=inp["logit_offset"],
                     capacity_factor=wl.capacity_factor,
                     n_groups=wl.n_groups, topk_groups=wl.topk_groups,
                     group_score_topk=wl.group_score_topk, device=device)
    torch.cuda.synchronize()
    return layer, inp


def launches_per_step(layer, routed):
    from combine_router_gemm_top_b300 import _lib as L
    # layout (one block, or histogram + scan + assignment), permute, combine
    n = L.moe_dispatch_layout_launches(layer.T, layer.k, layer.E) + 1 + 1
    if routed:
        # route: one kernel up to 32 experts (moe_route_launches says when),
        # else the router GEMM and the select kernel
        n += L.moe_route_launches(layer.cfg)
    if not layer.identity:
        # grouped FFN: one launch, except fp32 with F > 12288 (up, down)
        n += 2 if ffn_variant(layer) == 4 else 1
    return n


def kernel_models(wl, n_kept, es, peaks, active_experts=None, t_kept=None):
    """Algorithmic work of each step and the roofline time it implies.
    Bytes count each input read once and each output written once;
    intermediates (split-K partial logits, the SwiGLU activations H) are not
    algorithmic.  t_kept: tokens with at least one kept pair, the rows
    permute reads (T when nothing is dropped)."""
    T, D, E, k, F = wl.T, wl.D, wl.E, wl.k, wl.F
    P, N = T * k, n_kept
    Tk = T if t_kept is None else t_kept
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops_sustained"] * 1e12
    m = {}
    m["route"] = dict(bytes=T * D * es + E * D * es + P * 8,
                      flops=2.0 * T * D * E)
    m["layout"] = dict(bytes=P * 4 + P * 4 + N * 4, flops=0.0)
    m["permute"] = dict(bytes=Tk * D * es + N * D * es + P * 4, flops=0.0)
    if not wl.identity_experts:
        ea = E if active_experts is None else active_experts
        m["ffn"] = dict(bytes=ea * 3 * F * D * es + 2 * N * D * es,
                        flops=6.0 * D * F * N)
    m["combine"] = dict(bytes=N * D * es + T * D * es + P * 8, flops=0.0)
    for v in m.values():
        t_hbm = v["bytes"] / hbm
        t_tc = v["flops"] / tc if wl.dtype == "bf16" else 0.0
        v["bound"] = "tensor" if t_tc > t_hbm else "hbm"
        v["roofline_ms"] = max(t_hbm, t_tc) * 1e3
    return m


def tokens_kept(layer):
    """Tokens with at least one kept pair: the x rows moe_permute reads
    (counted after the timed region, from the layout's dst_row)."""
    dst = layer.dst_row[:layer.T * layer.k].view(layer.T, layer.k)
    return int((dst >= 0).any(dim=1).sum().item())


def replica_seed(base_seed, rank):
    """Each replica draws its own batch: weak scaling, no shared data."""
    return base_seed + rank


def max_over_ranks(value, device, dist=None):
    """The slowest replica's time (the job finishes when it does); the
    value itself with one process."""
    import torch
    if dist is None or not dist.is_initialized():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# the configurations measured beside the headline workload, each as a
# sub-record of the default run's line
SUB_WORKLOADS = ("deepseek_bf16", "switch_bf16", "tiny_f32",
                 "sweep_bf16_uniform_T65536", "sweep_bf16_zipf_T65536")
STAGES = ["route", "layout", "permute", "ffn", "combine"]


def ffn_variant(layer):
    from combine_router_gemm_top_b300 import _lib as L
    return L.moe_grouped_ffn_variant(layer.E, layer.D, layer.F,
                                     layer.T * layer.k, layer.dcode)


def kernel_label(layer, key):
    from combine_router_gemm_top_b300 import _lib as L
    n_layout = L.moe_dispatch_layout_launches(layer.T, layer.k, layer.E)
    return {
        "ffn": {1: "moe_grouped_ffn (fp32: one CUDA-core launch, a block "
                   "per row)",
                4: "moe_grouped_ffn (fp32: up and down kernels on CUDA cores)",
                2: "moe_grouped_ffn (one tcgen05 launch, up + down, one SM "
                   "per 128-row tile)",
                3: "moe_grouped_ffn (one tcgen05 launch, up + down, SM pairs "
                   "on 256-row tiles)"}.get(ffn_variant(layer),
                                            "moe_grouped_ffn"),
        "route": (("moe_route (one kernel: 16-token tiles on the warp-level "
                   "MMA)" if layer.cfg.dtype == L.MOE_BF16 else
                   "moe_route (one warp-per-token kernel)")
                  if L.moe_route_launches(layer.cfg) == 1 else
                  "moe_route (router GEMM + select)"),
        "layout": f"moe_dispatch_layout ({n_layout} launch"
                  f"{'es' if n_layout > 1 else ''})",
        "permute": "moe_permute", "combine": "moe_combine"}[key]


def measure(args, wl, dev, rank, world, local_rank, dist):
    """Times K steps of one workload (every stage, from the step graphs) and
    returns (record, layer, inp, extra) where record holds the throughput,
    the per-kernel rooflines and the clocks."""
    import torch
    layer, inp = build_layer(wl, dev, replica_seed(wl.seed, rank))
    x = inp["x"]
    idx_in = inp.get("topk_idx")      # pre-drawn routing (sweep workloads)
    gate_in = inp.get("topk_gate")
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stages = [lambda s: layer.route(x, s),
              lambda s: layer.dispatch_layout(idx_in, s),
              lambda s: layer.permute(x, s),
              lambda s: layer.grouped_ffn(s),
              lambda s: layer.combine(gate_in, None, s)]
    for _ in range(args.warmup):
        flush.zero_()
        for fn in stages:
            fn(stream)
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()}")
    graphs = capture_step_graphs(stages, flush, dev)
    run_step_graphs(graphs, GRAPH_RING)
    K = args.steps
    clocks = ClockSampler(local_rank)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.5)
    t_wall0 = time.perf_counter()
    times = run_step_graphs(graphs, K)
    wall = time.perf_counter() - t_wall0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    del graphs
    parts = {key: sum(t[j] for t in times) for j, key in enumerate(STAGES)}
    total_ms = max_over_ranks(sum(parts.values()), dev, dist)
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    n_kept = int(layer.n_kept.item())
    active = int((layer.expert_counts > 0).sum().item())
    es = x.element_size()
    peaks = load_peaks()
    tc_peak, tc_note = choose_bf16_peak(peaks, wall, clk)
    models = kernel_models(wl, n_kept, es, peaks, active, tokens_kept(layer))
    kernels = {}
    for key, mdl in models.items():
        ms = parts[key] / K
        if mdl["bound"] == "tensor":
            ach, unit, pk = mdl["flops"] / (ms / 1e3) / 1e12, "TFLOP/s", \
                tc_peak
        else:
            ach, unit, pk = mdl["bytes"] / (ms / 1e3) / 1e9, "GB/s", \
                peaks["hbm_gbs"]
        kernels[key] = {"ms": round(ms, 4), "bound": mdl["bound"],
                        "achieved": round(ach, 1), "unit": unit,
                        "frac": round(ach / pk, 4),
                        "roofline_ms": round(mdl["roofline_ms"], 4)}
        if mdl["flops"] and wl.dtype == "bf16":
            kernels[key]["tflops"] = round(mdl["flops"] / (ms / 1e3) / 1e12, 1)
    dom = max(kernels, key=lambda kk: kernels[kk]["ms"])
    dk, dm = kernels[dom], models[dom]
    if dk["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dk["achieved"],
                "peak": tc_peak, "unit": "TFLOP/s", "frac": dk["frac"],
                "traffic": None, "peak_note": tc_note,
                "frac_of_burst": round(dk["achieved"] / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(
                    dk["achieved"] / peaks["bf16_tflops_sustained"], 4),
                "algorithmic_per_launch": dm["flops"]}
    else:
        roof = {"bound": "hbm", "achieved": dk["achieved"],
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dk["frac"],
                "traffic": None, "peak_note": "HBM copy, " + peaks["source"],
                "algorithmic_per_launch": dm["bytes"]}
    # DRAM bytes (read + write) of one launch of the dominant kernel, from an
    # ncu capture of the same kernel on the same workload; re-take it when
    # the kernel changes.
    dram = NCU_DRAM_BYTES.get((wl.name, wl.T, wl.E, dom, ffn_variant(layer)))
    if dram is not None:
        roof["traffic"] = dram
        roof["traffic_over_algorithmic"] = round(dram / dm["bytes"], 3)
    roof["kernel"] = kernel_label(layer, dom)
    pc_bytes = models["permute"]["bytes"] + models["combine"]["bytes"]
    pc_ms = (parts["permute"] + parts["combine"]) / K
    pc_gbs = pc_bytes / (pc_ms / 1e3) / 1e9
    rec = {
        "value": round(wl.T * world * K / (total_ms / 1e3), 1),
        "unit": "tokens/s", "ms_per_step": round(total_ms / K, 4),
        "steps": K,
        "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E,
                   "k": wl.k, "F": wl.F, "R": wl.R,
                   "capacity": layer.capacity or "dropless",
                   "score": wl.score, "dtype": wl.dtype, "n_kept": n_kept,
                   "active_experts": active,
                   "routing": wl.routing or "router"},
        "kernels": kernels,
        "permute_combine": {"gbs": round(pc_gbs, 1),
                            "frac_of_hbm": round(pc_gbs / peaks["hbm_gbs"], 4),
                            "algorithmic_bytes": pc_bytes},
        "roofline": roof,
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3)}
    extra = dict(x=x, idx_in=idx_in, gate_in=gate_in, flush=flush,
                 stream=stream, es=es)
    return rec, layer, inp, extra


def run_ours(args, rank, world, local_rank, workload=None, cpu=True,
             subs=()):
    import torch
    from combine_router_gemm_top_b300 import workloads as W
    dist = None
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.WORKLOADS[workload or args.workload]
    if args.tokens:
        wl = wl.with_(T=args.tokens)
    if args.experts:
        wl = wl.with_(E=args.experts, R=min(wl.R, args.experts))
    rec, layer, inp, ex = measure(args, wl, dev, rank, world, local_rank,
                                  dist)
    x, idx_in, gate_in = ex["x"], ex["idx_in"], ex["gate_in"]
    stream, flush, es = ex["stream"], ex["flush"], ex["es"]
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    # end to end through the public layer API from pinned host memory: a
    # stream of batches, each copied in, run and copied out; copies of the
    # neighbouring batches overlap the compute (MoELayer.forward_host_stream).
    # The per-step working set (weights plus activations) exceeds L2.
    ring = 4
    xs_host = [x.cpu().pin_memory() for _ in range(ring)]
    ys_host = [torch.empty_like(layer.y, device="cpu").pin_memory()
               for _ in range(ring)]
    e2e_steps = max(4, min(args.steps, 200))
    xs = [xs_host[i % ring] for i in range(e2e_steps)]
    ys = [ys_host[i % ring] for i in range(e2e_steps)]
    layer.forward_host_stream(xs[:ring], ys[:ring], stream, idx_in, gate_in)
    torch.cuda.synchronize()
    a_ev, b_ev = ev(), ev()
    a_ev.record(stream)
    layer.forward_host_stream(xs, ys, stream, idx_in, gate_in)
    b_ev.record(stream)
    b_ev.synchronize()
    e2e_ms = max_over_ranks(a_ev.elapsed_time(b_ev), dev, dist)

    # the same step replayed as one CUDA graph through MoELayer.capture
    replay = layer.capture(x, idx_in, gate_in)
    for _ in range(3):
        replay()
    g_steps = max(3, min(K_graph_cap, args.steps))
    g_ms = 0.0
    for _ in range(g_steps):
        flush.zero_()
        a_ev, b_ev = ev(), ev()
        a_ev.record(stream)
        replay()
        b_ev.record(stream)
        b_ev.synchronize()
        g_ms += a_ev.elapsed_time(b_ev)
    g_ms = max_over_ranks(g_ms, dev, dist)
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()}")
    launches = launches_per_step(layer, True) * args.steps
    cpu_line = None
    if rank == 0 and world == 1 and cpu and not args.no_cpu_baseline:
        # the oracle on the host cores, fed the same (device) inputs
        cpu_line = run_cpu_baseline(wl, inp)
    del layer, inp, flush, ex, replay
    torch.cuda.empty_cache()

    # the other configurations, each measured the same way
    sub_recs = {}
    for name in subs:
        if name == wl.name:
            continue
        r, lay, inp2, ex2 = measure(args, W.WORKLOADS[name], dev, rank,
                                    world, local_rank, dist)
        sub_recs[name] = r
        del lay, inp2, ex2
        torch.cuda.empty_cache()
    if rank != 0:
        return None

    K = args.steps
    e2e_tokens_s = wl.T * world * e2e_steps / (e2e_ms / 1e3)
    cfg = dict(rec["config"])
    cfg.update({"parallelism": f"replicas x{world}",
                "l2": "flushed (256 MiB write) before every timed step",
                "launch": "each step one CUDA graph with timing events "
                          "between its stages: stage times are device time"})
    line = {
        "metric": METRIC, "value": rec["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; random-init weights of the stated "
                "shapes)",
        "config": cfg,
        "kernels": rec["kernels"],
        "permute_combine": rec["permute_combine"],
        "roofline": rec["roofline"],
        "e2e": {"value": round(e2e_tokens_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.T * wl.D * es,
                "d2h_bytes_per_step": wl.T * wl.D * es,
                "steps": e2e_steps,
                "how": "MoELayer.forward_host_stream: pinned host x in and "
                       "y out every step, copies of neighbouring steps "
                       "overlapping compute"},
        "graph": {"ms_per_step": round(g_ms / g_steps, 4),
                  "tokens_per_s": round(wl.T * world * g_steps /
                                        (g_ms / 1e3), 1),
                  "steps": g_steps,
                  "how": "MoELayer.capture: the whole step as one CUDA "
                         "graph, L2 flushed before every replay"},
        "gpu_launches": launches,
        "clocks": rec["clocks"],
        "wall_s_timed_loop": rec["wall_s_timed_loop"],
    }
    if sub_recs:
        line["workloads"] = sub_recs
    line["cpu_baseline"] = cpu_line
    return line


# ------------------------------------------------------- beyond the step
def run_extras(args, local_rank, workload):
    """Times the calls outside the five-step layer pass on one workload:
    router statistics (L_aux, f, P), the bias step, the kept-pair dispatch
    matrix and, for capacity workloads, the padded static-capacity path
    (padded layout, pad fill, permute, grouped FFN and combine on E*C rows).
    Each call is timed alone with CUDA events, after an L2 flush, median of
    the repeats.  One JSON line per workload."""
    import torch
    from combine_router_gemm_top_b300 import _lib as L
    from combine_router_gemm_top_b300 import workloads as W
    from combine_router_gemm_top_b300.layer import MoELayer
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.WORKLOADS[workload]
    inp = W.make_inputs(wl, device=dev, seed=wl.seed)
    layer = MoELayer(wl.T, wl.D, wl.E, wl.k, wl.R, inp["w_r"], inp["w13"],
                     inp["w2"], F=wl.F, score=wl.score,
                     sel_bias=inp["sel_bias"],
                     logit_offset=inp["logit_offset"],
                     capacity_factor=wl.capacity_factor,
                     n_groups=wl.n_groups, topk_groups=wl.topk_groups,
                     group_score_topk=wl.group_score_topk, device=dev,
                     keep_logits=True)
    x = inp["x"]
    layer.forward(x)
    torch.cuda.synchronize()
    peaks = load_peaks()
    hbm = peaks["hbm_gbs"]
    T, D, E, k, P = wl.T, wl.D, wl.E, wl.k, wl.T * wl.k
    es = x.element_size()
    n_kept = int(layer.n_kept.item())
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    reps = max(5, min(args.steps, 50))

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            host_ahead()
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    i32 = dict(dtype=torch.int32, device=dev)
    out = {}

    def put(name, ms, nbytes=None, flops=None):
        d = {"ms": round(ms, 4)}
        if nbytes is not None:
            gbs = nbytes / (ms / 1e3) / 1e9
            d.update(bytes=nbytes, gbs=round(gbs, 1), bound="hbm",
                     frac_of_hbm=round(gbs / hbm, 4))
        if flops is not None:
            tf = flops / (ms / 1e3) / 1e12
            d.update(flops=flops, tflops=round(tf, 1), bound="tensor",
                     frac_of_sustained=round(
                         tf / peaks["bf16_tflops_sustained"], 4))
        out[name] = d

    st = torch.zeros(1, **i32)
    ws = torch.empty(L.moe_router_stats_workspace_size(T, E),
                     dtype=torch.uint8, device=dev)
    f = torch.empty(E, dtype=torch.float32, device=dev)
    Pm = torch.empty(E, dtype=torch.float32, device=dev)
    cnt = torch.empty(E, **i32)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    put("router_stats", timed(lambda: L.moe_router_stats(
        T, E, k, wl.score, layer.logits, layer.topk_idx, 0.01, f, Pm, cnt,
        loss, ws, st)), nbytes=T * E * 4 + P * 4)
    bias = torch.zeros(E, dtype=torch.float32, device=dev)
    put("router_bias_update", timed(lambda: L.moe_router_bias_update(
        T, k, E, cnt, 1e-3, bias)), nbytes=E * 12)
    R = wl.R
    mat = torch.empty(R * R, **i32)
    put("dispatch_matrix", timed(lambda: L.moe_dispatch_matrix(
        T, k, E, R, R, layer.topk_idx, layer.dst_row, mat, st)),
        nbytes=2 * P * 4)
    # micro-batches: four batches of T tokens one after another, and the
    # same four with the routing, layout and permute of batch i+1 on a
    # second stream while batch i's experts (on all SMs but 8) and combine
    # run (MoELayer.forward_overlapped)
    if not layer.identity:
        n_mb = 4
        xs = [x] * n_mb
        ys = [torch.empty_like(x) for _ in range(n_mb)]

        def sequential():
            for xi, yi in zip(xs, ys):
                layer.forward(xi, y=yi)
        layer.forward_overlapped(xs, ys)      # builds the twin buffers
        put("microbatches_sequential", timed(sequential))
        put("microbatches_overlapped",
            timed(lambda: layer.forward_overlapped(xs, ys)))
        out["microbatches_overlapped"]["gain_vs_sequential"] = round(
            out["microbatches_sequential"]["ms"] /
            out["microbatches_overlapped"]["ms"] - 1.0, 4)
    cap = layer.capacity
    if cap > 0 and not layer.identity:
        rows = E * cap
        dst_p = torch.empty(P, **i32)
        off_p = torch.empty(E + 1, **i32)
        xpad = torch.empty((rows, D), dtype=x.dtype, device=dev)
        ypad = torch.empty_like(xpad)
        fws = torch.empty(L.moe_grouped_ffn_workspace_size(
            E, D, wl.F, rows, layer.dcode), dtype=torch.uint8, device=dev)
        y = torch.empty_like(x)
        put("padded_layout", timed(lambda: L.moe_padded_layout(
            T, k, E, cap, layer.topk_idx, layer.dst_row,
            layer.expert_offsets, dst_p, off_p, st)), nbytes=3 * P * 4)
        put("pad_fill", timed(lambda: L.moe_pad_fill(
            E, cap, D, layer.dcode, layer.expert_counts, xpad)),
            nbytes=(rows - n_kept) * D * es)
        put("padded_permute", timed(lambda: L.moe_permute(
            T, k, D, layer.dcode, x, dst_p, xpad, layer.status)),
            nbytes=tokens_kept(layer) * D * es + n_kept * D * es + P * 4)
        put("padded_ffn", timed(lambda: L.moe_grouped_ffn(
            E, D, wl.F, rows, layer.dcode, xpad, off_p, layer.w13, layer.w2,
            ypad, fws, st)), flops=6.0 * D * wl.F * rows)
        put("padded_combine", timed(lambda: L.moe_combine(
            T, k, D, layer.dcode, ypad, dst_p, layer.topk_gate, y,
            layer.status)),
            nbytes=n_kept * D * es + T * D * es + P * 8)
    torch.cuda.synchronize()
    if st.item() != 0 or layer.device_status() != 0:
        raise RuntimeError("device status set during the extras")
    line = {"mode": "extras", "workload": wl.name,
            "config": {"T": T, "D": D, "E": E, "k": k, "F": wl.F, "R": R,
                       "capacity": cap or "dropless", "n_kept": n_kept},
            "repeats": reps, "timing": "CUDA events per call, L2 flushed, "
                                       "median",
            "peaks": {"hbm_gbs": hbm,
                      "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                      "source": peaks["source"]},
            "kernels": out}
    del layer, inp, flush
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------- training step
def run_train(args, local_rank, workload):
    """One training step of the layer: forward on the 64-row aligned layout
    (forward_train) then the backward pass, timed with CUDA events per
    stage, L2 flushed before every step.  The expert backward (five tcgen05
    GEMMs) is reported against the sustained bf16 peak with its useful
    FLOPs 16*N*D*F (dH 2, recomputed gate/up 4, dXp 4, dW2 2, dW13 4)."""
    import torch
    from combine_router_gemm_top_b300 import workloads as W
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.WORKLOADS[workload]
    if args.tokens:
        wl = wl.with_(T=args.tokens)
    if args.experts:
        wl = wl.with_(E=args.experts, R=min(wl.R, args.experts))
    layer, inp = build_layer(wl, dev, wl.seed)
    x = inp["x"]
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 17)
    dy = torch.randn(x.shape, generator=g, device=dev).to(x.dtype)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    from combine_router_gemm_top_b300 import _lib as L
    b = layer._train_buffers()
    names = ["forward", "combine_bwd", "ffn_bwd", "permute_bwd", "route_bwd"]

    def step(m=None):
        rec = (lambda j: m[j].record(stream)) if m else (lambda j: None)
        rec(0)
        layer.forward_train(x, stream)
        rec(1)
        L.moe_combine_backward(wl.T, wl.k, wl.D, layer.dcode, dy, b["ya"],
                               b["dst_a"], layer.topk_gate, b["dga"],
                               b["dgate"], layer.status, stream)
        L.moe_aligned_fill(wl.E, wl.D, layer.dcode, layer.expert_offsets,
                           b["off_a"], b["dga"], stream)
        rec(2)
        L.moe_grouped_ffn_backward(wl.E, wl.D, wl.F, b["rows"], layer.dcode,
                                   b["xa"], b["dga"], b["off_a"], layer.w13,
                                   layer.w2, b["dxa"], b["dw13"], b["dw2"],
                                   b["bwd_ws"], layer.status, stream)
        rec(3)
        L.moe_permute_backward(wl.T, wl.k, wl.D, layer.dcode, b["dxa"],
                               b["dst_a"], b["dx"], layer.status, stream)
        rec(4)
        L.moe_route_backward(layer.cfg, x, layer.w_r, layer.logits,
                             layer.topk_idx, b["dgate"], b["dlogits"],
                             b["dw_r"], b["dx"], b["route_bwd_ws"],
                             layer.status, stream)
        rec(5)

    layer._x = x
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    K = max(1, min(args.steps, 200))
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    marks = [[ev() for _ in range(6)] for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.5)
    for i in range(K):
        flush.zero_()
        step(marks[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()}")
    parts = {n: sum(m[j].elapsed_time(m[j + 1]) for m in marks) / K
             for j, n in enumerate(names)}
    total = sum(m[0].elapsed_time(m[5]) for m in marks) / K
    peaks = load_peaks()
    n_kept = int(layer.n_kept.item())
    flops_bwd = 16.0 * n_kept * wl.D * wl.F
    flops_fwd = 6.0 * n_kept * wl.D * wl.F
    tf_bwd = flops_bwd / (parts["ffn_bwd"] / 1e3) / 1e12
    line = {"mode": "train", "metric": "MoE-layer training-step tokens/s "
                                       "(forward + backward) at 1 B300",
            "value": round(wl.T / (total / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(total, 4), "steps": K,
            "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E,
                       "k": wl.k, "F": wl.F, "n_kept": n_kept,
                       "aligned_rows": int(b["off_a"][-1].item()),
                       "l2": "flushed (256 MiB write) before every step"},
            "per_stage_ms": {n: round(v, 4) for n, v in parts.items()},
            "ffn_backward": {"tflops": round(tf_bwd, 1),
                             "frac_of_sustained": round(
                                 tf_bwd / peaks["bf16_tflops_sustained"], 4),
                             "useful_flops": flops_bwd},
            "forward_train_tflops": round(
                flops_fwd / (parts["forward"] / 1e3) / 1e12, 1),
            "clocks": clk}
    del layer, inp, flush
    torch.cuda.empty_cache()
    return line


# --------------------------------------------------------------- CPU oracle
def oracle_sample_run(wl, inp, n_tok):
    """One pass of the CPU oracle (as it stands) over the first n_tok tokens
    of the workload; returns seconds."""
    import numpy as np
    import torch
    import oracle.moe_oracle as O

    def f64(t):
        return t.detach().to("cpu", torch.float64).numpy()

    class Lazy:
        # expert weights converted to float64 when the oracle reads them
        def __init__(self, t):
            self.t = t

        def __getitem__(self, e):
            return f64(self.t[e])

    t0 = time.perf_counter()
    x = f64(inp["x"][:n_tok])
    cap = O.expert_capacity(wl.capacity_factor, n_tok, wl.k, wl.E)
    if wl.routing is not None:
        O.moe_forward(x, None, wl.k, wl.E, wl.R, wl.score,
                      topk_idx=inp["topk_idx"][:n_tok].cpu().numpy(),
                      topk_gate=f64(inp["topk_gate"][:n_tok]))
    else:
        O.moe_forward(
            x, f64(inp["w_r"]), wl.k, wl.E, wl.R, wl.score,
            w13=Lazy(inp["w13"]), w2=Lazy(inp["w2"]),
            sel_bias=None if inp["sel_bias"] is None
            else inp["sel_bias"].cpu().numpy(),
            logit_offset=None if inp["logit_offset"] is None
            else inp["logit_offset"].cpu().numpy(),
            n_groups=wl.n_groups, topk_groups=wl.topk_groups,
            group_score_topk=wl.group_score_topk, capacity=cap)
    return time.perf_counter() - t0


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info()
             if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def cpu_inputs(wl):
    from combine_router_gemm_top_b300 import workloads as W
    return W.make_inputs(wl, device="cpu")


def run_cpu_baseline(wl, inp, steps=1):
    n_tok = min(wl.T, CPU_SAMPLE_TOKENS.get(wl.name, 256))
    secs = [oracle_sample_run(wl, inp, n_tok) for _ in range(steps)]
    s = sum(secs) / len(secs)
    return {"value": round(n_tok / s, 3), "unit": "tokens/s",
            "cores": cpu_threads(), "kind": "oracle",
            "sample": f"first {n_tok} of {wl.T} tokens of {wl.name} "
                      f"(full route, layout, permute, fp64 experts, "
                      f"combine), {s:.1f} s per pass"}


REF_BUDGET_S = 150.0   # bound on the reference arm's timed work


def run_reference(args, rank, world):
    """The CPU oracle as it stands, on the host cores: each step is one
    oracle pass over a bounded token sample of the workload.  If K such
    steps would run past REF_BUDGET_S, only as many as fit are timed
    (reported as steps_timed)."""
    if rank != 0:
        return None
    from combine_router_gemm_top_b300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    inp = cpu_inputs(wl)
    n_tok = min(wl.T, REF_SAMPLE_TOKENS.get(wl.name, 64))
    first = oracle_sample_run(wl, inp, n_tok)          # warm-up pass
    steps = max(1, min(args.steps, int(REF_BUDGET_S / max(first, 1e-3))))
    secs = [oracle_sample_run(wl, inp, n_tok) for _ in range(steps)]
    total = sum(secs)
    value = n_tok * steps / total
    cb = {"value": round(value, 3), "unit": "tokens/s",
          "cores": cpu_threads(), "kind": "oracle",
          "sample": f"first {n_tok} of {wl.T} tokens of {wl.name} per step "
                    f"(route, layout, permute, fp64 experts, combine)"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "steps_timed": steps, "warmup": args.warmup,
            "ms_per_step": round(total / steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E,
                       "k": wl.k, "F": wl.F, "sample_tokens": n_tok},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 3), "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="mixtral_bf16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (small cases "
                         "for profiler captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the workload's expert count (small cases "
                         "for profiler captures)")
    ap.add_argument("--train", action="store_true",
                    help="time one training step (forward on the aligned "
                         "layout + backward) of --workload")
    ap.add_argument("--extras", action="store_true",
                    help="time router statistics, the bias step, the "
                         "dispatch matrix and the padded static-capacity "
                         "path: one JSON line per workload")
    ap.add_argument("--only", action="store_true",
                    help="measure --workload alone (no sub-records of the "
                         "other configurations)")
    ap.add_argument("--sweep", action="store_true",
                    help="dispatch/combine bandwidth sweep: one JSON line "
                         "per (T, routing) identity-expert workload")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        from combine_router_gemm_top_b300 import build as B
        if rank == 0:
            B.build(verbose=False)
        if args.train:
            if rank == 0:
                print(json.dumps(run_train(args, local_rank, args.workload)),
                      flush=True)
            return
        if args.extras:
            if rank == 0:
                for name in ("switch_bf16", "deepseek_bf16", "mixtral_bf16",
                             "tiny_f32"):
                    print(json.dumps(run_extras(args, local_rank, name)),
                          flush=True)
            return
        if args.sweep:
            for T in (4096, 16384, 65536):
                for r in ("uniform", "zipf"):
                    ln = run_ours(args, rank, world, local_rank,
                                  workload=f"sweep_bf16_{r}_T{T}", cpu=False)
                    if ln is not None:
                        print(json.dumps(ln), flush=True)
            return
        subs = () if (args.only or args.tokens or args.experts) else \
            SUB_WORKLOADS
        line = run_ours(args, rank, world, local_rank, subs=subs)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
