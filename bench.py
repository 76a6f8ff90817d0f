"""Benchmark of the routed + shared-expert MoE layer forward on GB300.

Default: one GPU, the Olmo-shaped bf16 layer (T=8192, d=2560, N=32 experts of
width 2560, top-4, one shared expert of width 1280), synthetic seeded inputs.
Prints ONE JSON line.  ``--impl reference`` times the CPU oracle instead (on
bounded samples of the same workload).  Under torchrun each rank runs its own
replica on its own batch (weak scaling, no collective on the data path); rank 0
prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import csv
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s and TFLOP/s (% of BF16 peak) on 1 GB300"
NOMINAL_HBM_GBS = 8000.0


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            m = json.load(fh)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    return p


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for r in csv.reader(fh):
                if len(r) >= 9:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- oracle timing

def time_oracle(spec, inp_host, budget_s: float, min_tokens: int = 64):
    """Run the oracle on the first S tokens of the workload; S sized for ~budget_s seconds."""
    import oracle as O

    def run(S):
        sub = spec.replace(T=S)
        d = dict(inp_host)
        d["x"] = inp_host["x"][:S]
        t0 = time.perf_counter()
        O.moe_forward(sub, d)
        return time.perf_counter() - t0

    S = min(min_tokens, spec.T)
    t = run(S)
    while t < budget_s / 4 and S < spec.T:
        S = min(spec.T, max(S * 2, int(S * budget_s / max(t, 1e-3) / 2)))
        t = run(S)
    return S, t


# ----------------------------------------------------------------- entropy sweep

def histograms(N: int, R: int):
    """Kept-count histograms over N experts with R routes in total (fixed work).

    Families: uniform; one hot expert holding a share s of the routes ("spike");
    three hot experts sharing s ("three-hot"), the rest spread evenly.  Pairs of
    spike / three-hot histograms with the same maximum load are included.
    """
    def spread(hot):
        rest = R - sum(hot)
        k = N - len(hot)
        base = [rest // k + (1 if i < rest % k else 0) for i in range(k)]
        return hot + base
    out = [("uniform", spread([]))]
    for s in (0.1, 0.2, 0.3, 0.45, 0.6, 0.8):
        out.append((f"spike s={s}", spread([int(R * s)])))
        out.append((f"three-hot s={s}", spread([int(R * s / 3)] * 3)))
    # same maximum load as the spike with share s: three experts at that load
    for s in (0.1, 0.2, 0.3):
        m = int(R * s)
        out.append((f"three-hot max={m}", spread([m, m, m])))
    return out


def entropy_deficit(counts):
    import math
    tot = float(sum(counts))
    H = -sum((c / tot) * math.log(c / tot) for c in counts if c > 0)
    return 1.0 - H / math.log(len(counts))


def sweep_entropy(args, spec):
    """Grouped-GEMM throughput vs the kept-count entropy deficit at fixed total work
    (Section 10.2's fixed-work microbenchmark of local expert compute)."""
    import torch
    import routing_shared_expert_gb300 as moe
    from workloads import make_inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = make_inputs(spec, dev)
    cfg = moe.config_from_spec(spec)
    ws = moe.alloc_workspace(cfg, dev)
    R = spec.T * spec.K
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    x_perm = torch.randn((R, spec.d_model), generator=g, device=dev).to(spec.torch_dtype)
    f = torch.empty((R, spec.d_model), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flops = 6.0 * spec.d_model * spec.d_expert * R
    rows = []
    for name, counts in histograms(spec.N, R):
        assert sum(counts) == R and len(counts) == spec.N
        offs = torch.tensor([0] + list(__import__("itertools").accumulate(counts)), dtype=torch.int32, device=dev)
        for _ in range(3):
            moe.moe_grouped_swiglu(cfg, x_perm, offs, None, inp["W_gate"], inp["W_up"], inp["W_down"], f, ws)
        torch.cuda.synchronize()
        ms = 0.0
        for _ in range(args.steps):
            flush.add_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            moe.moe_grouped_swiglu(cfg, x_perm, offs, None, inp["W_gate"], inp["W_up"], inp["W_down"], f, ws)
            b.record()
            torch.cuda.synchronize()
            ms += a.elapsed_time(b)
        ms /= args.steps
        rows.append({"histogram": name, "max_load": max(counts), "entropy_deficit": round(entropy_deficit(counts), 4),
                     "ms": round(ms, 4), "tflops": round(flops / ms / 1e9, 1)})
    assert moe.moe_read_status(ws) == 0
    base = rows[0]["tflops"]
    for r in rows:
        r["normalized"] = round(r["tflops"] / base, 4)
        print(json.dumps(r), flush=True)
    return 0


def launches_per_step(spec) -> int:
    """Kernels moe_layer_forward launches for a layer (counted from the library's launch
    sequence): router 1; permutation 4 (count, scan, place, row copy); routed experts 2;
    shared expert 2 or 0; combine 1."""
    return 1 + 4 + 2 + (2 if spec.d_shared > 0 else 0) + 1


# ----------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="olmo")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--sweep", choices=["entropy"], default=None,
                    help="instead of the benchmark line: grouped-GEMM throughput vs entropy deficit")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from workloads import CONFIGS, make_inputs
    spec = CONFIGS[args.config]
    if args.sweep == "entropy":
        return sweep_entropy(args, spec)
    cores = len(os.sched_getaffinity(0))
    config = {"workload": spec.name, "T": spec.T, "d_model": spec.d_model, "N": spec.N,
              "d_expert": spec.d_expert, "K": spec.K, "d_shared": spec.d_shared,
              "score": spec.score, "norm": spec.norm, "alpha": spec.alpha,
              "shared": spec.shared_mode, "capacity": spec.cap_policy}

    if args.impl == "reference":
        if rank != 0:
            return 0
        import torch
        inp = make_inputs(spec, "cpu")
        times, toks = [], 0
        for i in range(args.warmup + args.steps):
            S, t = time_oracle(spec, inp, budget_s=min(args.cpu_budget, 6.0), min_tokens=64)
            if i >= args.warmup:
                times.append(t)
                toks += S
        total = sum(times)
        val = toks / total
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(config, sample=f"first {S} tokens per step"),
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"first {S} of {spec.T} tokens of the {spec.name} layer per step"},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import routing_shared_expert_gb300 as moe
    inp = make_inputs(spec, dev, seed=0)
    if world > 1:
        # each rank its own batch of tokens (weak scaling); weights are the same replica
        inp["x"] = make_inputs(spec.replace(N=1, d_expert=64, d_shared=0), dev, seed=rank)["x"]
    layer = moe.MoELayer(moe.config_from_spec(spec), inp, dev)
    x = inp["x"]
    stream = torch.cuda.current_stream()

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        layer.forward(x, logits=False)
        flush.add_(1)
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # Timed region: the fused layer call a user makes (moe_layer_forward), with four events
    # recorded inside it by the library after router, permutation, routed experts and
    # shared expert + combine.
    stage_names = ("route", "permute", "grouped_swiglu", "shared_combine")
    stage_ms = {k: 0.0 for k in stage_names}
    step_ms = []
    for _ in range(args.steps):
        flush.add_(1)                        # write 256 MiB (> L2) between steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        layer.forward_profiled(x, ev)
        torch.cuda.synchronize()
        step_ms.append(ev[0].elapsed_time(ev[4]))
        for i, k in enumerate(stage_names):
            stage_ms[k] += ev[i].elapsed_time(ev[i + 1])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()

    # end to end through the public call: pinned host x -> device, forward, y -> pinned host
    x_host = x.cpu().pin_memory()
    y_host = torch.empty(layer.out["y"].shape, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x)
    e2e = []
    for _ in range(args.steps):
        flush.add_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        y = layer.forward(x_dev, logits=False)
        y_host.copy_(y, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        e2e.append(a.elapsed_time(b))

    total_ms = sum(step_ms)
    t_tensor = torch.tensor([total_ms, sum(e2e)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t_tensor, op=dist.ReduceOp.MAX)
    total_ms, e2e_ms = float(t_tensor[0]), float(t_tensor[1])

    assert layer.status() == 0, "device status word set during the benchmark"
    kept = int(layer.out["counts_keep"].sum())
    ms = total_ms / args.steps
    tokens_per_s = world * spec.T / (ms / 1e3)
    flops = spec.expert_flops(kept)
    tflops = world * flops / (ms / 1e3) / 1e12
    pk = peaks()
    g_ms = stage_ms["grouped_swiglu"] / args.steps
    g_flops = 6.0 * spec.d_model * spec.d_expert * kept
    g_tf = g_flops / (g_ms / 1e3) / 1e12

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
        "config": dict(config, l2="256 MiB buffer written between timed steps (flushes the 129 MB L2)",
                       timing="CUDA events on the launching stream around each moe_layer_forward call, "
                              "stage events recorded inside it"),
        "tflops": tflops, "pct_bf16_peak": 100.0 * tflops / pk["bf16_tflops"],
        "stages_ms": {k: v / args.steps for k, v in stage_ms.items()},
        "roofline": {"kernel": "grouped_swiglu stage (tcgen05 gate/up + down GEMM launches over packed segments)",
                     "bound": "tensor", "achieved": g_tf, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": g_tf / pk["bf16_tflops"],
                     "frac_sustained": g_tf / pk["bf16_tflops_sustained"],
                     "peak_source": pk["source"], "traffic": None},
        "e2e": {"value": world * spec.T / (e2e_ms / args.steps / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": layer.out["y"].numel() * 4},
        "gpu_launches": launches_per_step(spec) * args.steps,
        "clocks": clk,
        "kept_routes": kept,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hin = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
        S, t = time_oracle(spec, hin, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": S / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {S} of {spec.T} tokens of the {spec.name} layer, "
                                          f"full forward in float64 ({t:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
