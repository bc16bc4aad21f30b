"""Benchmark of the MoE-layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one whole layer pass (route -> dispatch layout -> permute ->
grouped SwiGLU FFN -> combine) over one batch of seeded synthetic input with
every input resident in HBM.  The default workload is the Mixtral-like
top-2 layer (T=2048, D=4096, E=8, k=2, F=14336, bf16, dropless).  Between
timed steps a 256 MiB buffer (> the 126 MB L2) is overwritten, outside the
timed events, so every step starts with a cold L2.

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


def launches_per_step(layer):
    n = 2 + 3 + 1 + 1            # route (GEMM + select), layout, permute, combine
    if not layer.identity:
        n += 2                   # grouped FFN: up and down projections
    return n


def run_ours(args, rank, world, local_rank):
    import torch
    from combine_router_gemm_top_b300 import workloads as W
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.WORKLOADS[args.workload]
    layer, inp = build_layer(wl, dev, wl.seed + rank)
    x = inp["x"]
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        layer.route(x, stream)
        layer.dispatch_layout(None, stream)
        layer.permute(x, stream)
        layer.grouped_ffn(stream)
        layer.combine(None, None, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError(f"device status {layer.device_status()}")

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    marks = [[ev() for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        m = marks[i]
        m[0].record(stream)
        layer.route(x, stream)
        m[1].record(stream)
        layer.dispatch_layout(None, stream)
        m[2].record(stream)
        layer.permute(x, stream)
        m[3].record(stream)
        layer.grouped_ffn(stream)
        m[4].record(stream)
        layer.combine(None, None, stream)
        m[5].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()

    parts = {"route": 0.0, "layout": 0.0, "permute": 0.0, "ffn": 0.0,
             "combine": 0.0}
    total_ms = 0.0
    for m in marks:
        for j, key in enumerate(parts):
            parts[key] += m[j].elapsed_time(m[j + 1])
        total_ms += m[0].elapsed_time(m[5])
    if dist is not None:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())

    # end to end through the public layer API from pinned host memory
    x_host = x.cpu().pin_memory()
    y_host = torch.empty_like(layer.y, device="cpu").pin_memory()
    x_dev = torch.empty_like(x)
    for _ in range(max(1, args.warmup)):
        flush.zero_()
        layer.forward_host(x_host, y_host, x_dev, stream)
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record(stream)
        layer.forward_host(x_host, y_host, x_dev, stream)
        b.record(stream)
        b.synchronize()
        e2e_ms += a.elapsed_time(b)
    if dist is not None:
        t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    n_kept = int(layer.n_kept.item())
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    K = args.steps
    es = x.element_size()
    peaks = load_peaks()
    tokens = wl.T * world * K
    value = tokens / (total_ms / 1e3)
    ms_step = total_ms / K
    pc_bytes = 2 * (wl.T * wl.D * es + n_kept * wl.D * es) + \
        wl.T * wl.k * (4 + 4 + 4)
    pc_ms = (parts["permute"] + parts["combine"]) / K
    pc_gbs = pc_bytes / (pc_ms / 1e3) / 1e9
    if layer.identity:
        dom = "permute+combine"
        achieved = pc_gbs
        roof = {"bound": "hbm", "kernel": "moe_permute+moe_combine",
                "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": None,
                "algorithmic_bytes_per_step": pc_bytes}
    else:
        dom = "moe_grouped_ffn"
        flops = 6.0 * wl.D * wl.F * n_kept
        ffn_ms = parts["ffn"] / K
        achieved = flops / (ffn_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if wl.dtype == "bf16" else None
        roof = {"bound": "tensor", "kernel": "moe_grouped_ffn (tcgen05 up + "
                "down launches)", "achieved": round(achieved, 2),
                "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4) if peak else None,
                "traffic": None, "peak_kind": "bf16 sustained, "
                + peaks["source"],
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                "algorithmic_flops_per_launch": flops}
    e2e_tokens_s = tokens / (e2e_ms / 1e3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; random-init weights of the stated "
                "shapes)",
        "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E,
                   "k": wl.k, "F": wl.F, "R": wl.R,
                   "capacity": layer.capacity or "dropless",
                   "score": wl.score, "n_kept": n_kept,
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed (256 MiB write) before every timed step"},
        "per_step_ms": {k2: round(v / K, 4) for k2, v in parts.items()},
        "permute_combine": {"gbs": round(pc_gbs, 1),
                            "frac_of_hbm": round(pc_gbs / peaks["hbm_gbs"], 4),
                            "algorithmic_bytes": pc_bytes},
        "roofline": roof,
        "dominant_kernel": dom,
        "e2e": {"value": round(e2e_tokens_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.T * wl.D * es,
                "d2h_bytes_per_step": wl.T * wl.D * es},
        "gpu_launches": launches_per_step(layer) * K,
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3),
    }
    if dist is not None:
        dist.destroy_process_group()
    elif not args.no_cpu_baseline:
        # the oracle on the host cores, fed the same (device) inputs
        line["cpu_baseline"] = run_cpu_baseline(wl, inp)
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


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from combine_router_gemm_top_b300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    inp = cpu_inputs(wl)
    n_tok = min(wl.T, REF_SAMPLE_TOKENS.get(wl.name, 64))
    for _ in range(min(args.warmup, 1)):
        oracle_sample_run(wl, inp, min(n_tok, 8))
    secs = [oracle_sample_run(wl, inp, n_tok) for _ in range(args.steps)]
    total = sum(secs)
    value = n_tok * args.steps / total
    cb = {"value": round(value, 3), "unit": "tokens/s",
          "cores": cpu_threads(), "kind": "oracle",
          "sample": f"first {n_tok} of {wl.T} tokens of {wl.name} per step"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 1),
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixtral_bf16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        line = run_ours(args, rank, world, local_rank)
        if line is not None and "cpu_baseline" not in line:
            line["cpu_baseline"] = None
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
