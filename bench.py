"""Benchmark of the routed + shared-expert MoE layer forward on GB300.

Default: one GPU, the DeepSeek-V3-shaped bf16 layer (T=8192, d=7168, N=256 experts
of width 2048, top-8 sigmoid routing renormalised with alpha=2.5, one shared expert
of width 2048), the largest of the benchmark layers, synthetic seeded inputs.  The
Olmo-, Qwen2- and Mixtral-shaped layers are timed the same way and reported in the
line's ``per_config`` block.  Prints ONE JSON line.  ``--impl reference`` times the
CPU oracle instead (on bounded samples of the same workload).  Under torchrun each
rank runs its own replica on its own batch (weak scaling, no collective on the data
path); rank 0 prints the line with the max time over ranks.
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


# DRAM traffic of the dominant stage (the routed gate/up and down launches of one
# moe_grouped_swiglu call), dram__bytes_read.sum + dram__bytes_write.sum summed over the
# two launches, from one ncu capture per workload.  It is reported only while the kernel
# sources hash to the value they had at capture time.
STAGE_TRAFFIC = {"dsv3": {"sources_sha256": "6ca7eee779d4d719", "bytes": 29247472896}}
TRAFFIC_SOURCES = ("routing_shared_expert_gb300/csrc/gemm_tc2.cu", "routing_shared_expert_gb300/csrc/common.cuh")


def stage_traffic(name: str):
    import hashlib
    rec = STAGE_TRAFFIC.get(name)
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sources_sha256"] else None


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
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "power.draw.instant")

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
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float = None, t1: float = None):
        """Summarise the samples taken between wall-clock times t0 and t1 (the timed
        region); if none fell inside it, the samples nearest to it are used instead."""
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
                if len(r) >= 10:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        return summarize_clocks(rows, t0, t1)


def _stamp(text: str):
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(text, fmt).timestamp()
        except ValueError:
            pass
    return None


def summarize_clocks(rows, t0=None, t1=None):
    """rows: nvidia-smi CSV records (timestamp, index, sm, max sm, power, active, four reasons,
    and optionally the instantaneous power).  power.draw is a one-second average, which in a
    timed region of a fraction of a second still reads mostly the idle time before it; the
    instantaneous reading follows the load."""
    if not rows:
        return None
    stamped = [(_stamp(r[0]), r) for r in rows]
    inside = [r for t, r in stamped if t is not None and t0 is not None and t0 <= t <= t1]
    window = "timed region"
    if not inside and t0 is not None:
        near = sorted((abs(t - 0.5 * (t0 + t1)), i) for i, (t, _) in enumerate(stamped) if t is not None)
        inside = [stamped[i][1] for _, i in near[:2]]
        window = "nearest samples (timed region shorter than the sampling interval)"
    if not inside:
        inside, window = rows, "whole run"

    def num(v):
        try:
            return float(v)
        except ValueError:
            return None

    sm = [v for v in (num(r[2]) for r in inside) if v is not None]
    mx = [v for v in (num(r[3]) for r in inside) if v is not None]
    pw = [v for v in (num(r[4]) for r in inside) if v is not None]
    pi = [v for v in (num(r[10]) for r in inside if len(r) > 10) if v is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "power_w": statistics.median(pw) if pw else None,
            "power_instant_w": statistics.median(pi) if pi else None,
            "power_instant_max_w": max(pi) if pi else None,
            "reasons": reasons, "samples": len(inside), "window": window}


def max_over_ranks(values, device, world: int):
    """Each rank's totals -> the element-wise maximum over ranks (the slowest rank sets
    the job's time)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return world * tokens_per_rank * steps / (total_ms / 1e3)


# ----------------------------------------------------------------- oracle timing

class ExpertsF64:
    """Per-expert float64 host copies of a [N, ...] weight tensor (on the device or the
    host), converted on first use and kept up to a host-memory cap: the oracle's inputs held
    resident in its own number format, as the GPU arm's are held resident in HBM.  The
    conversion is input preparation, so timed oracle runs are repeated (at most twice)
    while they convert; weights beyond the cap are converted inside the timed run, and the
    count of such conversions is reported with the sample."""

    CAP_BYTES = 8 << 30
    held = 0            # bytes cached over all instances
    conversions = 0     # conversions so far (a timed run must add none)

    def __init__(self, t):
        self.t, self.cache = t, {}

    def __getitem__(self, e):
        if e in self.cache:
            return self.cache[e]
        import oracle as O
        a = O.f64(self.t[e])
        ExpertsF64.conversions += 1
        if ExpertsF64.held + a.nbytes <= ExpertsF64.CAP_BYTES:
            self.cache[e] = a
            ExpertsF64.held += a.nbytes
        return a


def oracle_inputs(inp_host: dict) -> dict:
    import oracle as O
    out = {}
    for k, v in inp_host.items():
        if k in ("W_gate", "W_up", "W_down"):
            out[k] = ExpertsF64(v)
        elif hasattr(v, "detach") and v.is_floating_point():
            out[k] = O.f64(v)
        else:
            out[k] = v
    return out


def oracle_seconds(spec, inp_host, S: int) -> float:
    """Wall time of the oracle's full layer forward on the first S tokens, its weights
    already converted where they fit the cache: the run is repeated, at most twice more,
    while it converted weights that the cache kept (conversions past the cache's cap recur
    on every run, so a repeat would not remove them); ``oracle_seconds.converted`` holds the
    last run's conversions."""
    sub = spec.replace(T=S)
    d = dict(inp_host)
    d["x"] = inp_host["x"][:S]
    import oracle as O
    for _ in range(3):
        c0, h0 = ExpertsF64.conversions, ExpertsF64.held
        t0 = time.perf_counter()
        O.moe_forward(sub, d)
        t = time.perf_counter() - t0
        oracle_seconds.converted = ExpertsF64.conversions - c0
        if oracle_seconds.converted == 0 or ExpertsF64.held == h0:
            break
    return t


oracle_seconds.converted = 0


def time_oracle(spec, inp_host, budget_s: float, min_tokens: int = 64, max_sizes: int = 5):
    """Run the oracle on the first S tokens of the workload, S grown (at least doubling, aimed
    at budget_s) until one run takes three quarters of budget_s or covers every token, trying
    at most ``max_sizes`` sizes.  The run time need not grow in proportion to S: a few tokens
    already touch most experts, whose weights the oracle converts to float64."""
    S = min(min_tokens, spec.T)
    t = oracle_seconds(spec, inp_host, S)
    sizes = 1
    while t < 0.75 * budget_s and S < spec.T and sizes < max_sizes:
        S = min(spec.T, max(S * 2, int(S * budget_s / max(t, 1e-3))))
        t = oracle_seconds(spec, inp_host, S)
        sizes += 1
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
    W_down = moe.pack_weights(inp["W_down"]) if cfg.h_format == 1 else inp["W_down"]
    R = spec.T * spec.K
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    x_perm = torch.randn((R, spec.d_model), generator=g, device=dev).to(spec.torch_dtype)
    f = torch.empty((R, spec.d_model), dtype=torch.float16 if cfg.h_format == 1 else torch.float32,
                    device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flops = 6.0 * spec.d_model * spec.d_expert * R
    rows = []
    for name, counts in histograms(spec.N, R):
        assert sum(counts) == R and len(counts) == spec.N
        offs = torch.tensor([0] + list(__import__("itertools").accumulate(counts)), dtype=torch.int32, device=dev)
        for _ in range(3):
            moe.moe_grouped_swiglu(cfg, x_perm, offs, None, inp["W_gate"], inp["W_up"], W_down, f, ws)
        torch.cuda.synchronize()
        ms = 0.0
        for _ in range(args.steps):
            flush.add_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            moe.moe_grouped_swiglu(cfg, x_perm, offs, None, inp["W_gate"], inp["W_up"], W_down, f, ws)
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


def stage_algorithmic_bytes(spec, kept: int) -> int:
    """Bytes the grouped stage must move at least once: packed rows x_perm and the routed
    weights (gate, up, down) read, h written and read, f written (fp16 for bf16 layers,
    whose intermediate format is fp16; fp32 for fp32 layers)."""
    b = spec.elem_bytes
    d, dr, N = spec.d_model, spec.d_expert, spec.N
    return int(kept * d * b + 3 * N * d * dr * b + 2 * kept * dr * b + kept * d * b)


def stage_roofline(spec, kept: int, g_ms: float, pk) -> dict:
    """The grouped stage against the roof that binds it.  Its algorithmic intensity (routed
    expert FLOP over the stage's algorithmic bytes) against the measured ridge (bf16 peak over
    HBM rate) decides: below the ridge the stage is bound by HBM and is measured in GB/s,
    above it by the tensor cores in TFLOP/s.  Both fractions are reported."""
    flops = 6.0 * spec.d_model * spec.d_expert * kept
    nbytes = stage_algorithmic_bytes(spec, kept)
    sec = g_ms / 1e3
    ai = flops / nbytes
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    tf = flops / sec / 1e12
    gbs = nbytes / sec / 1e9
    out = {"intensity_flop_per_byte": ai, "ridge_flop_per_byte": ridge,
           "frac_tensor": tf / pk["bf16_tflops"], "frac_hbm": gbs / pk["hbm_gbs"]}
    if ai < ridge:
        out.update({"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / pk["hbm_gbs"]})
    else:
        out.update({"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": tf / pk["bf16_tflops"],
                    "frac_sustained": tf / pk["bf16_tflops_sustained"]})
    return out


def layer_algorithmic_bytes(spec, kept: int) -> int:
    """Bytes one layer forward must move at least once, summed over its steps: the router
    (x and W_router read, top-K written), the permutation (top-K read, route tables written,
    x read, x_perm written), the grouped stage (stage_algorithmic_bytes), the shared expert
    (x and its weights read, its intermediate written and read, g written) and the combine
    (f, g and the route tables read, fp32 y written).  Intermediates h, f and g take the
    layer's element size (fp16 for bf16 layers, whose intermediate format is fp16)."""
    b = spec.elem_bytes
    T, d, N, K, ds = spec.T, spec.d_model, spec.N, spec.K, spec.d_shared
    routes = T * K
    router = T * d * b + N * d * b + 2 * routes * 4
    permute = routes * 4 + 2 * routes * 4 + T * d * b + kept * d * b
    shared = (T * d * b + 3 * d * ds * b + 2 * T * ds * b + T * d * b) if ds > 0 else 0
    combine = kept * d * b + (T * d * b if ds > 0 else 0) + T * d * 4 + 2 * routes * 4
    return int(router + permute + stage_algorithmic_bytes(spec, kept) + shared + combine)


def layer_roofline(spec, kept: int, ms: float, pk) -> dict:
    """The whole layer against its roofline: executed expert and shared FLOP over the layer's
    algorithmic bytes gives its intensity; the roof is the lower of the bf16 peak and
    intensity x HBM rate (both measured), and frac is the achieved FLOP rate over that roof."""
    flops = spec.expert_flops(kept)
    nbytes = layer_algorithmic_bytes(spec, kept)
    ai = flops / nbytes
    roof = min(pk["bf16_tflops"], ai * pk["hbm_gbs"] / 1e3)
    tf = flops / (ms / 1e3) / 1e12
    return {"flops": flops, "bytes": nbytes, "intensity_flop_per_byte": ai,
            "ridge_flop_per_byte": pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"],
            "bound": "tensor" if roof >= pk["bf16_tflops"] else "hbm",
            "roof_tflops": roof, "achieved_tflops": tf, "frac": tf / roof}


def experts_window(spec, kept: int, stage_ms: dict, world: int, pk) -> dict:
    """All expert GEMM FLOP (routed and shared) over the window they run in: from the start
    of the layer to the end of the routed experts (the router, the permutation and the
    routed experts on the caller's stream; the shared expert beside them on the second
    stream).  The grouped stage alone counts only routed FLOP while a large shared expert's
    tail runs inside it."""
    ms = stage_ms["route"] + stage_ms["permute"] + stage_ms["grouped_swiglu"]
    tf = world * spec.expert_flops(kept) / (ms / 1e3) / 1e12
    return {"ms": ms, "tflops": tf, "frac_tensor": tf / pk["bf16_tflops"]}


def launches_per_step(spec, sms: int = 152) -> int:
    """Kernels moe_layer_forward launches for a layer (counted from the library's launch
    sequence): router 1; permutation 2 (counting, capacity and placement in one launch while
    the 256-token tiles fit on the GPU at once, which holds here for up to one tile per SM,
    else 3; then the row copy); routed experts 2; shared expert 2 or 0; combine 1."""
    permute = 2 if (spec.T + 255) // 256 <= sms else 4
    return 1 + permute + 2 + (2 if spec.d_shared > 0 else 0) + 1


# ----------------------------------------------------------------- balance
def bench_balance(args, spec, config, dev) -> int:
    """The load-balancing side outputs of one routed batch (moe_balance_stats: P, f and the
    statistics of Eq. 22, 27, 30 and 39 and the entropy deficit) and one bias-controller step
    (moe_bias_update, Eq. 37): three launches, timed together per call with CUDA events
    (queued behind a device-side wait, so the interval excludes host launch cost), L2
    flushed between calls, on the routing of the workload's own router and permutation.  They read only the
    routing (logits [T][N] fp32 and the counts), so the expert widths are reduced to keep
    the device footprint small."""
    import torch
    import routing_shared_expert_gb300 as moe
    from routing_shared_expert_gb300 import _native as nat
    from workloads import make_inputs
    sp = spec.replace(d_expert=128, d_shared=128 if spec.d_shared else 0)
    inp = make_inputs(sp, dev, seed=0)
    layer = moe.MoELayer(moe.config_from_spec(sp), inp, dev)
    layer.forward(inp["x"], logits=True)
    o, c, ws = layer.out, layer.cfg, layer.ws
    f32 = dict(dtype=torch.float32, device=dev)
    P, f, stats = torch.empty(sp.N, **f32), torch.empty(sp.N, **f32), torch.empty(len(nat.STATS), **f32)
    bias = torch.zeros(sp.N, **f32)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        nat.moe_balance_stats(c, o["logits"], o["counts_req"], o["counts_keep"], o["R_req"],
                              o["R_keep"], P, f, stats, ws)
        nat.moe_bias_update(sp.N, o["counts_req"], 1e-3, bias)

    times = []
    for i in range(args.warmup + args.steps):
        flush.add_(1)
        # a device-side wait ahead of the start event, so that the three launches are queued
        # before the GPU reaches it and the interval holds device time only
        torch.cuda._sleep(2_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e3)
    if layer.status() != 0:
        raise RuntimeError(f"layer status {layer.status()}")
    us = statistics.median(times)
    M = sp.num_ranks
    nbytes = sp.T * sp.N * 4 + 2 * sp.N * 4 + 2 * M * 4 + 2 * sp.N * 4 + len(nat.STATS) * 4 + 2 * sp.N * 4
    pk = peaks()
    gbs = nbytes / (us / 1e6) / 1e9
    print(json.dumps({"mode": "balance", "workload": spec.name, "us_per_call": us,
                      "calls": args.steps, "gpu_launches_per_call": 3, "algorithmic_bytes": nbytes,
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                                   "unit": "GB/s", "frac": gbs / pk["hbm_gbs"]},
                      "stats": {k: float(v) for k, v in zip(nat.STATS, stats.cpu().tolist())},
                      "config": dict(config, note="expert widths reduced to 128 (the statistics "
                                                  "read only the routing)")}), flush=True)
    return 0


# ----------------------------------------------------------------- expert parallelism
def bench_ep(args, spec, config, dev) -> int:
    """The device side of one rank's expert-parallel forward (F4: Section 10.3, Figure 41) for
    the layout rho(i) = i mod M with M = the workload's rank count, on this GPU: the plan
    (moe_ep_keep_matrix, moe_ep_place, moe_ep_send_pos: three launches), the dispatch's two
    indexed row copies (the rank's x rows into its send buffer; a received buffer into its
    packed expert buffer by moe_ep_recv_rows) and the return's two (the packed outputs into
    the send-back buffer; the received outputs into one row per route, dropped routes zero).
    The all-to-all between them needs a second GPU and is not run: the other M - 1 sources
    are emulated with this rank's own request counts, so the buffers have the sizes of M
    equal sources.  CUDA events around each step, L2 flushed before each; bytes are the
    rows each copy must read and write once.  The expert widths are reduced (the exchange
    moves d_model-wide rows only)."""
    import torch
    import routing_shared_expert_gb300 as moe
    from routing_shared_expert_gb300 import _native as nat
    from routing_shared_expert_gb300 import ep
    from workloads import make_inputs
    sp = spec.replace(d_expert=128, d_shared=128 if spec.d_shared else 0)
    inp = make_inputs(sp, dev, seed=0)
    layer = moe.MoELayer(moe.config_from_spec(sp), inp, dev, staged_buffers=False)
    layer.forward(inp["x"], logits=False)
    c, o, ws = layer.cfg, layer.out, layer.ws
    T, K, N, d, M = sp.T, sp.K, sp.N, sp.d_model, max(sp.num_ranks, 1)
    rho = [e % M for e in range(N)]
    x = inp["x"]
    eb = x.element_size()
    # this rank's requests and its capacity-free permutation (the stable ranks moe_ep_place reads)
    i32 = dict(dtype=torch.int32, device=dev)
    cnt, ck, off = torch.empty(N, **i32), torch.empty(N, **i32), torch.empty(N + 1, **i32)
    rpos, psrc = torch.empty((T, K), **i32), torch.empty(T * K, **i32)
    free = moe.config_from_spec(sp.replace(cap_policy="none"))
    moe.moe_permute(free, None, o["topk_idx"], cnt, ck, off, rpos, psrc, None, None, None, None, ws)
    counts_all = cnt.unsqueeze(0).repeat(M, 1).contiguous()
    policy = sp.cap_policy if sp.cap_policy != "per_expert" else "rank_wide"
    rank = 0

    pl = ep.make_plan(counts_all, o["topk_idx"], rank, K, rho, policy, sp.capacity_factor,
                      route_pos=rpos, offsets=off, workspace=ws)
    lib = nat.library()
    rho_arr = ep._rho(rho)
    pol = nat.CAP_POLICIES[policy]
    keep, roff = torch.empty_like(pl.keep), torch.empty_like(pl.recv_off)
    rq, rk = torch.empty_like(pl.R_req), torch.empty_like(pl.R_keep)
    dst, spos = torch.empty_like(pl.dst_row), torch.empty_like(pl.send_pos)
    P = ep._ptr

    def plan():
        # the three device entries of the plan, without the host read of the keep matrix that
        # ep.make_plan adds for the all-to-all's split sizes
        st = nat._stream(None)
        nat._check("moe_ep_keep_matrix", lib.moe_ep_keep_matrix(
            M, N, K, rho_arr, pol, float(sp.capacity_factor), P(counts_all), P(keep), P(roff),
            P(rq), P(rk), st))
        nat._check("moe_ep_place", lib.moe_ep_place(
            M, rank, T, N, K, P(o["topk_idx"]), P(rpos), P(off), P(keep), P(roff), P(dst), P(ws),
            ws.numel(), st))
        nat._check("moe_ep_send_pos", lib.moe_ep_send_pos(
            M, rank, T, N, K, rho_arr, P(o["topk_idx"]), P(keep), P(roff), P(dst), P(spos), None,
            P(ws), ws.numel(), st))

    split = pl.send_counts()
    n_send = int(split[rank].sum())
    n_recv = int(split[:, rank].sum())
    n_local = int(pl.R_keep[rank])
    send = torch.empty((max(n_send, 1), d), dtype=x.dtype, device=dev)
    recv = torch.empty((max(n_recv, 1), d), dtype=x.dtype, device=dev).normal_()
    rows = torch.empty((max(n_local, 1), d), dtype=x.dtype, device=dev)
    back = torch.empty((max(n_send, 1), d), dtype=x.dtype, device=dev).normal_()
    out = torch.empty((T * K, d), dtype=x.dtype, device=dev)
    rr = ep.recv_rows(pl, workspace=ws)
    send_back = torch.empty((max(n_recv, 1), d), dtype=x.dtype, device=dev)
    steps = {
        "plan: keep matrix": (None, 3 * M * N * 4),
        "plan (keep matrix, destination rows, send positions)":
            (plan, T * K * 4 * 5 + 2 * M * N * 4),
        "dispatch: receive rows (moe_ep_recv_rows)":
            (lambda: nat._check("moe_ep_recv_rows", lib.moe_ep_recv_rows(
                M, rank, N, rho_arr, P(keep), P(roff), P(rr), rr.numel(), P(ws), ws.numel(),
                nat._stream(None))), n_recv * 4 + 2 * M * N * 4),
        "dispatch: x rows into the send buffer":
            (lambda: ep.rows_copy(x, send, T * K, src_div=K, dst_index=pl.send_pos, workspace=ws),
             T * d * eb + n_send * d * eb),
        "dispatch: received rows into the packed expert buffer":
            (lambda: ep.rows_copy(recv, rows, n_recv, dst_index=rr, workspace=ws),
             2 * n_recv * d * eb),
        "return: packed outputs into the send-back buffer":
            (lambda: ep.rows_copy(rows, send_back, n_recv, src_index=rr, workspace=ws),
             2 * n_recv * d * eb),
        "return: received outputs into one row per route (dropped routes zero)":
            (lambda: ep.rows_copy(back, out, T * K, src_index=pl.send_pos, zero_missing=True,
                                  workspace=ws),
             n_send * d * eb + T * K * d * eb),
    }
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    pk = peaks()
    results = {}
    def keep_only():
        nat._check("moe_ep_keep_matrix", lib.moe_ep_keep_matrix(
            M, N, K, rho_arr, pol, float(sp.capacity_factor), P(counts_all), P(keep), P(roff),
            P(rq), P(rk), nat._stream(None)))

    steps["plan: keep matrix"] = (keep_only, steps["plan: keep matrix"][1])
    for name, (fn, nbytes) in steps.items():
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            flush.add_(1)
            torch.cuda._sleep(2_000_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(times)
        gbs = nbytes / (us / 1e6) / 1e9
        results[name] = {"us": us, "algorithmic_bytes": nbytes, "GB_s": gbs,
                         "frac_hbm": gbs / pk["hbm_gbs"]}
    if layer.status() != 0:
        raise RuntimeError(f"layer status {layer.status()}")
    print(json.dumps({"mode": "ep", "workload": spec.name, "ranks": M, "policy": policy,
                      "rows": {"send": n_send, "receive": n_recv, "packed": n_local},
                      "calls": args.steps, "steps": results, "hbm_peak_gbs": pk["hbm_gbs"],
                      "not_run": "the all-to-all between the dispatch's and the return's two copies "
                                 "(one GPU: the other sources are emulated)",
                      "config": dict(config, note="expert widths reduced to 128 (the exchange "
                                                  "moves d_model-wide rows only)")}), flush=True)
    return 0


# ----------------------------------------------------------------- backward

def bench_backward(args, spec, layer, x, config, dev):
    """Time moe_layer_backward (router coefficients fixed) on the routing of one forward
    call: CUDA events around each call, a 256 MiB buffer written between calls."""
    import torch
    layer.forward(x, logits=True)
    rg = bool(args.router_grad)
    g = torch.Generator(device="cpu").manual_seed(7)
    dy = torch.randn((spec.T, spec.d_model), generator=g).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        layer.backward(x, dy, router_grad=rg)
        flush.add_(1)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    evs = []
    w0 = time.time()
    for _ in range(args.steps):
        flush.add_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        layer.backward(x, dy, router_grad=rg)
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop(w0, w1)
    assert layer.backward_status() == 0, "device status word set during the backward benchmark"
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    kept = int(layer.out["counts_keep"].sum())
    d, dr, ds = spec.d_model, spec.d_expert, spec.d_shared
    # per routed row: dgrad 6 d d_r, weight gradients 6 d d_r, recompute of a | b 4 d d_r
    std_flops = 12.0 * d * (dr * kept + ds * spec.T)
    exe_flops = 16.0 * d * (dr * kept + ds * spec.T)
    pk = peaks()
    line = {"metric": "MoE-layer backward (%s) tokens/s on 1 GB300" % (
                "including the router gradient" if rg else "router coefficients fixed"),
            "value": spec.T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": spec.dtype,
            "data": "synthetic", "config": dict(config, l2="256 MiB buffer written between calls"),
            "tflops_executed": exe_flops / (ms / 1e3) / 1e12,
            "tflops_standard": std_flops / (ms / 1e3) / 1e12,
            "pct_bf16_peak_executed": 100.0 * exe_flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"],
            "clocks": clk, "kept_routes": kept}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- main

def time_forward(spec, args, dev, world: int, rank: int, flush, stream, clocks_on: bool = True):
    """Warm up, then time args.steps moe_layer_forward calls of one layer (the fused call a
    user makes), with four events recorded inside each by the library after router,
    permutation, routed experts and combine (the shared expert runs on the library's second
    stream beside the first three; the last interval holds the wait for it and the combine).
    The steps are queued back to back (no host sync between them); a 256 MiB buffer is
    written between a step's last event and the next step's first (flushes the 129 MB L2).
    Returns the layer, its inputs and the timings (max over ranks)."""
    import torch
    import routing_shared_expert_gb300 as moe
    from workloads import make_inputs
    inp = make_inputs(spec, dev, seed=0)
    if world > 1:
        # each rank its own batch of tokens (weak scaling); weights are the same replica
        inp["x"] = make_inputs(spec.replace(N=1, d_expert=64, d_shared=0), dev, seed=rank)["x"]
    layer = moe.MoELayer(moe.config_from_spec(spec), inp, dev)
    x = inp["x"]
    for _ in range(max(args.warmup, 3)):
        layer.forward(x, logits=False)
        flush.add_(1)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device()) if clocks_on else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    stage_names = ("route", "permute", "grouped_swiglu", "join_combine")
    stage_ms = {k: 0.0 for k in stage_names}
    events = []
    w0 = time.time()
    for _ in range(args.steps):
        flush.add_(1)                        # write 256 MiB (> L2) between steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        layer.forward_profiled(x, ev, stream)
        events.append(ev)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clk = clocks.stop(w0, w1) if clocks else None
    step_ms = 0.0
    for ev in events:
        step_ms += ev[0].elapsed_time(ev[4])
        for i, k in enumerate(stage_names):
            stage_ms[k] += ev[i].elapsed_time(ev[i + 1])
    vals = max_over_ranks([step_ms] + [stage_ms[k] for k in stage_names], dev, world)
    assert layer.status() == 0, f"device status word set while timing {spec.name}"
    kept = int(layer.out["counts_keep"].sum())
    return {"layer": layer, "inp": inp, "x": x, "total_ms": vals[0],
            "stage_ms": {k: v / args.steps for k, v in zip(stage_names, vals[1:])},
            "clocks": clk, "kept": kept}


def summarize(spec, r, args, world: int, pk):
    """Throughput, executed TFLOP/s and the grouped stage's roofline of one timed layer."""
    kept = r["kept"]
    ms = r["total_ms"] / args.steps
    flops = spec.expert_flops(kept)
    tflops = world * flops / (ms / 1e3) / 1e12
    g_ms = r["stage_ms"]["grouped_swiglu"]
    g_tf = 6.0 * spec.d_model * spec.d_expert * kept / (g_ms / 1e3) / 1e12
    return {"ms_per_step": ms, "tokens_per_s": job_tokens_per_s(world, spec.T, args.steps, r["total_ms"]),
            "tflops": tflops, "pct_bf16_peak": 100.0 * tflops / pk["bf16_tflops"],
            "grouped_tflops": g_tf, "grouped_frac": g_tf / pk["bf16_tflops"],
            "grouped_roofline": stage_roofline(spec, kept, g_ms, pk),
            "experts_window": experts_window(spec, kept, r["stage_ms"], world, pk),
            "layer_roofline": layer_roofline(spec, kept, ms, pk),
            "stages_ms": r["stage_ms"], "kept_routes": kept}


def workload_config(spec):
    return {"workload": spec.name, "T": spec.T, "d_model": spec.d_model, "N": spec.N,
            "d_expert": spec.d_expert, "K": spec.K, "d_shared": spec.d_shared,
            "score": spec.score, "norm": spec.norm, "alpha": spec.alpha,
            "shared": spec.shared_mode, "capacity": spec.cap_policy,
            "intermediate": ("h, f and g fp16; down projections packed to fp16 once "
                             "(moe_pack_weights); fp32 accumulation" if spec.dtype == "bf16" else "fp32")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="dsv3")
    ap.add_argument("--per-config", default="olmo,qwen2,mixtral",
                    help="other workloads timed the same way and reported in per_config ('none': skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--sweep", choices=["entropy"], default=None,
                    help="instead of the benchmark line: grouped-GEMM throughput vs entropy deficit")
    ap.add_argument("--override", default="", metavar="K=V,...",
                    help="change integer fields of the workload (e.g. N=32,T=1024: a smaller layer "
                         "of the same shape per expert, for profiler captures)")
    ap.add_argument("--mode", choices=["forward", "backward", "balance", "ep"], default="forward",
                    help="backward: time moe_layer_backward (router coefficients fixed) on the "
                         "routing of one forward call, instead of the forward benchmark line; "
                         "balance: time the load-balancing statistics and the bias-controller step; "
                         "ep: time the device side of one rank's expert-parallel exchange")
    ap.add_argument("--router-grad", action="store_true",
                    help="with --mode backward: include the gradient through the router coefficients")
    ap.add_argument("--forward-only", type=int, default=0, metavar="R",
                    help="run R untimed layer forwards and exit (a short, fixed launch sequence "
                         "for ncu captures: each forward launches the routed gate/up and down "
                         "GEMMs, then the shared ones)")
    ap.add_argument("--route-only", type=int, default=0, metavar="R",
                    help="run R untimed router calls (moe_route alone) on the workload's inputs "
                         "and exit (the launch sequence of a router capture)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from workloads import CONFIGS, make_inputs
    spec = CONFIGS[args.config]
    if args.override:
        spec = spec.replace(**{k: int(v) for k, v in (kv.split("=") for kv in args.override.split(","))})
    if args.sweep == "entropy":
        return sweep_entropy(args, spec)
    cores = len(os.sched_getaffinity(0))
    config = workload_config(spec)

    if args.impl == "reference":
        if rank != 0:
            return 0
        import torch
        # the same seeded tensors as the GPU arm (drawn on the device when there is one,
        # then read by the oracle on the host cores)
        src = "cuda" if torch.cuda.is_available() else "cpu"
        inp = oracle_inputs(make_inputs(spec, src))
        # one bounded sample size S for every step, sized so the whole run takes a few minutes
        per_step = min(args.cpu_budget, max(0.05, 150.0 / (args.warmup + args.steps)))
        S, _ = time_oracle(spec, inp, budget_s=per_step, min_tokens=16)
        times, toks = [], 0
        for i in range(args.warmup + args.steps):
            t = oracle_seconds(spec, inp, S)
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
    if args.route_only > 0:
        inp = make_inputs(spec, dev, seed=0)
        layer = moe.MoELayer(moe.config_from_spec(spec), inp, dev, staged_buffers=False)
        c, o, w = layer.cfg, layer.out, layer.weights
        for _ in range(args.route_only):
            moe.moe_route(c, inp["x"], w["W_router"], w.get("router_bias"), w.get("selection_bias"),
                          w.get("shared_gate_w"), o["topk_idx"], o["topk_w"], o["shared_coef"], None,
                          layer.ws)
        torch.cuda.synchronize()
        if layer.status() != 0:
            raise RuntimeError(f"layer status {layer.status()}")
        print(json.dumps({"route_only": args.route_only, "workload": spec.name}), flush=True)
        return 0
    if args.forward_only > 0:
        inp = make_inputs(spec, dev, seed=0)
        layer = moe.MoELayer(moe.config_from_spec(spec), inp, dev)
        for _ in range(args.forward_only):
            layer.forward(inp["x"], logits=False)
        torch.cuda.synchronize()
        if layer.status() != 0:
            raise RuntimeError(f"layer status {layer.status()}")
        print(json.dumps({"forward_only": args.forward_only, "workload": spec.name,
                          "kept": int(layer.out["counts_keep"].sum())}), flush=True)
        return 0
    stream = torch.cuda.current_stream()
    if args.mode == "backward":
        inp = make_inputs(spec, dev, seed=0)
        layer = moe.MoELayer(moe.config_from_spec(spec), inp, dev)
        return bench_backward(args, spec, layer, inp["x"], config, dev)
    if args.mode == "balance":
        return bench_balance(args, spec, config, dev)
    if args.mode == "ep":
        return bench_ep(args, spec, config, dev)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    pk = peaks()
    r = time_forward(spec, args, dev, world, rank, flush, stream)
    layer, inp, x = r["layer"], r["inp"], r["x"]
    head = summarize(spec, r, args, world, pk)
    head_clocks = r["clocks"]

    # End to end through the public call: every step copies its x from pinned host memory,
    # runs moe_layer_forward and copies y back to pinned host memory, all inside the timed
    # region.  The copies run on their own streams, so step i's copy-out and step i+1's
    # copy-in overlap step i+1's / step i's compute (x and y double buffered).  No L2
    # flush here: as in a user's loop, each step reads all of the layer's weights (far
    # larger than L2) and an x freshly copied from the host.
    import routing_shared_expert_gb300._native as nat
    weight_bytes = sum(v.numel() * v.element_size() for k, v in inp.items()
                       if torch.is_tensor(v) and k != "x")
    x_host = x.cpu().pin_memory()
    y_host = [torch.empty(layer.out["y"].shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [torch.empty_like(layer.out["y"]) for _ in range(2)]
    base = {k: v for k, v in layer.out.items() if k not in ("logits", "y")}
    outs = [nat.make_outputs(y=y_dev[i], **base) for i in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(args.steps)]
    ev_fwd = [torch.cuda.Event() for _ in range(args.steps)]
    ev_out = [torch.cuda.Event() for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record(s_in)
    for i in range(args.steps):
        j = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_fwd[i - 2])        # x buffer j read by forward i-2
            x_dev[j].copy_(x_host, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])          # y buffer j read by copy-out i-2
        nat.moe_layer_forward(layer.cfg, layer.w, x_dev[j], outs[j], layer.ws, stream)
        ev_fwd[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_fwd[i])
            y_host[j].copy_(y_dev[j], non_blocking=True)
            ev_out[i].record(s_out)
    s_out.wait_event(ev_out[args.steps - 1])
    t_b.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([t_a.elapsed_time(t_b)], dev, world)[0]
    assert torch.equal(y_host[(args.steps - 1) % 2], layer.forward(x, logits=False).cpu()), \
        "end-to-end result differs from the device result"
    assert layer.status() == 0, "device status word set during the benchmark"
    kept = head["kept_routes"]
    e2e = {"value": job_tokens_per_s(world, spec.T, args.steps, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": x.numel() * x.element_size(),
           "d2h_bytes_per_step": layer.out["y"].numel() * 4,
           "method": "pinned host x -> device, moe_layer_forward, y -> pinned host every step; "
                     "copies on their own streams overlap the neighbouring steps' compute",
           "l2": f"no flush: every step reads {weight_bytes / 1e9:.2f} GB of weights (> L2) "
                 "and a freshly copied x"}

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle reads each expert's weights from the device copy and converts it to
        # float64 on first use (held up to the cache's cap)
        hin = oracle_inputs(inp)
        S, t = time_oracle(spec, hin, budget_s=args.cpu_budget)
        conv = oracle_seconds.converted
        cpu_baseline = {"value": S / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                        "sample": f"first {S} of {spec.T} tokens of the {spec.name} layer, "
                                  f"full forward in float64 ({t:.1f} s"
                                  + (f", including {conv} expert weight conversions to float64 "
                                     "that did not fit the 8 GB host cache)" if conv else ")")}
        del hin
    del layer, inp, x, r, x_host, y_host, x_dev, y_dev, outs
    torch.cuda.empty_cache()

    # the other bf16 workloads, each timed the same way (same steps, warm-up, L2 flush)
    per_config = {}
    names = [] if args.per_config in ("", "none") else args.per_config.split(",")
    for name in names:
        if name == spec.name or name not in CONFIGS:
            continue
        sp = CONFIGS[name]
        rr = time_forward(sp, args, dev, world, rank, flush, stream)
        sm = summarize(sp, rr, args, world, pk)
        clk = rr["clocks"] or {}
        per_config[name] = {"ms_per_step": sm["ms_per_step"], "tokens_per_s": sm["tokens_per_s"],
                            "tflops": sm["tflops"], "pct_bf16_peak": sm["pct_bf16_peak"],
                            "grouped_frac": sm["grouped_frac"],
                            "grouped_roofline": {k: sm["grouped_roofline"][k]
                                                 for k in ("bound", "frac", "frac_tensor", "frac_hbm")},
                            "experts_window": sm["experts_window"],
                            "layer_roofline": sm["layer_roofline"],
                            "stages_ms": sm["stages_ms"],
                            "kept_routes": sm["kept_routes"],
                            "clocks": {k: clk.get(k) for k in ("sm_mhz", "reasons", "samples")}}
        del rr
        torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic",
        "config": dict(config, l2="256 MiB buffer written between timed steps (flushes the 129 MB L2)",
                       timing="CUDA events on the launching stream around each moe_layer_forward call, "
                              "stage events recorded inside it"),
        "tflops": head["tflops"], "pct_bf16_peak": head["pct_bf16_peak"],
        "stages_ms": head["stages_ms"],
        "experts_window": head["experts_window"],
        "layer_roofline": head["layer_roofline"],
        "roofline": dict({"kernel": "grouped_swiglu stage (tcgen05 gate/up + down GEMM launches "
                                    "over packed segments)"},
                         **head["grouped_roofline"],
                         peak_source=pk["source"], traffic=stage_traffic(spec.name),
                         traffic_unit="bytes per stage (gate/up + down launches)",
                         algorithmic_bytes=stage_algorithmic_bytes(spec, kept)),
        "e2e": e2e,
        "gpu_launches": launches_per_step(
            spec, torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps,
        "clocks": head_clocks,
        "kept_routes": kept,
        "per_config": per_config,
    }
    if cpu_baseline is not None:
        line["cpu_baseline"] = cpu_baseline
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
