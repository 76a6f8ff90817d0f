"""Seeded synthetic workloads for the routed + shared-expert MoE layer forward.

This module is the one piece shared by the CUDA path (its tests and ``bench.py``)
and by the oracle's tests.  It only draws random numbers and lays them out in
the storage layout both sides read; it computes nothing of the layer itself
(no logits, no scores, no selection, no expert arithmetic).

Storage layout of one layer (row-major, the same on host and device):

* ``x``             [T, d]           token activations
* ``W_router``      [N, d]           one row per routed expert (logit z_ti = x_t . W_router[i])
* ``router_bias``   [N] fp32 or None additive per-expert logit bias
* ``shared_gate_w`` [d] or None      learned shared-branch gate vector w_s
* ``W_gate``        [N, d_r, d]      per expert, one row per intermediate unit (the columns of W_g)
* ``W_up``          [N, d_r, d]      same for W_u
* ``W_down``        [N, d, d_r]      per expert, one row per output dimension (the columns of W_d)
* ``Ws_gate``/``Ws_up`` [d_s, d], ``Ws_down`` [d, d_s]  the one (merged) shared expert, or None

The workload shapes are the five layer shapes of the benchmark table: a tiny
fp32 layer, and Olmo-, Qwen2-MoE-, DeepSeek-V3- and Mixtral-shaped bf16 layers.
Random numbers come from ``torch`` generators seeded per tensor (seed 0), drawn
on the device that will hold the tensor; the oracle always receives host
copies of exactly the tensors the device path consumed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int                 # tokens
    d_model: int           # d
    N: int                 # routed experts
    d_expert: int          # routed intermediate width d_r
    K: int                 # experts selected per token
    d_shared: int          # shared intermediate width d_s (0 = no shared expert)
    dtype: str             # "f32" or "bf16"
    score: str             # "softmax" | "sigmoid"
    norm: str              # "none" | "l1" | "softmax_selected" | "lp"
    alpha: float           # routed scale
    shared_mode: str       # "none" | "const" | "gate"
    shared_gain: float     # s when shared_mode == "const"
    cap_policy: str        # "none" | "per_expert" | "rank_wide"
    capacity_factor: float
    num_ranks: int         # M_E for the expert-to-rank map rho(i) = i mod M_E
    # input recipe
    init: str              # "fan_in" (std 1/sqrt(fan_in)) or "0.02" (std 0.02)
    logit_bias: str        # "none" | "normal" (N(0,1) per expert) | "zipf1.2"
    shared_split: tuple = ()   # widths of ungated shared experts that merge into d_shared
    norm_p: float = 2.0        # p of the "lp" rule

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    def rho(self):
        """Expert-to-rank map rho(i) = i mod M_E, as a list."""
        return [i % self.num_ranks for i in range(self.N)]

    def expert_flops(self, kept_routes: int) -> float:
        """Executed expert + shared GEMM FLOPs: 6 d (d_r R_keep + d_s T)."""
        return 6.0 * self.d_model * (self.d_expert * kept_routes + self.d_shared * self.T)


CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, d_model=64, N=8, d_expert=128, K=2, d_shared=64,
                      dtype="f32", score="softmax", norm="l1", alpha=2.0,
                      shared_mode="const", shared_gain=1.0, cap_policy="none",
                      capacity_factor=1.0, num_ranks=1, init="fan_in", logit_bias="none",
                      shared_split=(24, 24, 16)),
    "olmo": MoEConfig("olmo", T=8192, d_model=2560, N=32, d_expert=2560, K=4, d_shared=1280,
                      dtype="bf16", score="softmax", norm="l1", alpha=4.0,
                      shared_mode="const", shared_gain=1.0, cap_policy="none",
                      capacity_factor=1.0, num_ranks=1, init="0.02", logit_bias="none"),
    "qwen2": MoEConfig("qwen2", T=16384, d_model=2048, N=60, d_expert=1408, K=4, d_shared=5632,
                       dtype="bf16", score="softmax", norm="none", alpha=1.0,
                       shared_mode="gate", shared_gain=1.0, cap_policy="none",
                       capacity_factor=1.0, num_ranks=1, init="0.02", logit_bias="normal"),
    "dsv3": MoEConfig("dsv3", T=8192, d_model=7168, N=256, d_expert=2048, K=8, d_shared=2048,
                      dtype="bf16", score="sigmoid", norm="l1", alpha=2.5,
                      shared_mode="const", shared_gain=1.0, cap_policy="none",
                      capacity_factor=1.0, num_ranks=8, init="0.02", logit_bias="none"),
    "mixtral": MoEConfig("mixtral", T=32768, d_model=4096, N=8, d_expert=14336, K=2, d_shared=0,
                         dtype="bf16", score="softmax", norm="softmax_selected", alpha=1.0,
                         shared_mode="none", shared_gain=0.0, cap_policy="per_expert",
                         capacity_factor=1.0, num_ranks=1, init="0.02", logit_bias="zipf1.2"),
}

# Per-tensor seed offsets, so that each tensor's values do not depend on which
# other tensors were drawn first.
_TENSOR_IDS = {"x": 1, "W_router": 2, "router_bias": 3, "shared_gate_w": 4, "W_gate": 5,
               "W_up": 6, "W_down": 7, "Ws_gate": 8, "Ws_up": 9, "Ws_down": 10}


def _gen(device, seed: int, name: str, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + _TENSOR_IDS[name] * 10_007 + sub)
    return g


def _normal(shape, std: float, dtype, device, seed: int, name: str, sub: int = 0) -> torch.Tensor:
    g = _gen(device, seed, name, sub)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _std(cfg: MoEConfig, fan_in: int) -> float:
    return 1.0 / math.sqrt(fan_in) if cfg.init == "fan_in" else 0.02


def zipf_logit_bias(N: int, exponent: float = 1.2) -> torch.Tensor:
    """Per-expert logit bias b_i = -exponent * ln(i + 1).

    Adding it to the router logits scales the softmax odds of expert i by
    (i+1)^-exponent, a Zipf(exponent) popularity profile with expert 0 hottest.
    """
    return torch.tensor([-exponent * math.log(i + 1.0) for i in range(N)], dtype=torch.float32)


def make_inputs(cfg: MoEConfig, device="cpu", seed: int = 0,
                with_shared_parts: bool = False) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one layer's inputs and weights (see the module docstring for layout).

    Large per-expert tensors are drawn one expert at a time so that the fp32
    temporaries stay small.  With ``with_shared_parts`` and a config that names
    a shared split, the parts are also returned (``Ws_parts``: list of
    (gate, up, down)).  A config that names a split always draws its shared
    expert as those parts; the merged tensors are their plain concatenation
    (gate/up rows concatenated, down columns concatenated).
    """
    dev = torch.device(device)
    dt = cfg.torch_dtype
    T, d, N, dr, ds = cfg.T, cfg.d_model, cfg.N, cfg.d_expert, cfg.d_shared
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal((T, d), 1.0, dt, dev, seed, "x")
    out["W_router"] = _normal((N, d), _std(cfg, d), dt, dev, seed, "W_router")
    if cfg.logit_bias == "none":
        out["router_bias"] = None
    elif cfg.logit_bias == "normal":
        out["router_bias"] = _normal((N,), 1.0, torch.float32, dev, seed, "router_bias")
    elif cfg.logit_bias == "zipf1.2":
        out["router_bias"] = zipf_logit_bias(N, 1.2).to(dev)
    else:
        raise ValueError(cfg.logit_bias)
    out["shared_gate_w"] = (_normal((d,), 0.02 if cfg.init == "0.02" else _std(cfg, d), dt, dev,
                                    seed, "shared_gate_w")
                            if cfg.shared_mode == "gate" else None)

    W_gate = torch.empty((N, dr, d), dtype=dt, device=dev)
    W_up = torch.empty((N, dr, d), dtype=dt, device=dev)
    W_down = torch.empty((N, d, dr), dtype=dt, device=dev)
    for e in range(N):
        W_gate[e] = _normal((dr, d), _std(cfg, d), dt, dev, seed, "W_gate", e)
        W_up[e] = _normal((dr, d), _std(cfg, d), dt, dev, seed, "W_up", e)
        W_down[e] = _normal((d, dr), _std(cfg, dr), dt, dev, seed, "W_down", e)
    out["W_gate"], out["W_up"], out["W_down"] = W_gate, W_up, W_down

    if ds > 0:
        split = cfg.shared_split if cfg.shared_split else (ds,)
        assert sum(split) == ds
        parts = []
        for j, m in enumerate(split):
            # Each part is drawn at its own width; the init std of the down
            # projection uses the merged width d_s so that the merged expert
            # is one width-d_s expert of the recipe.
            pg = _normal((m, d), _std(cfg, d), dt, dev, seed, "Ws_gate", j)
            pu = _normal((m, d), _std(cfg, d), dt, dev, seed, "Ws_up", j)
            pd = _normal((d, m), _std(cfg, ds), dt, dev, seed, "Ws_down", j)
            parts.append((pg, pu, pd))
        out["Ws_gate"] = torch.cat([p[0] for p in parts], 0).contiguous()
        out["Ws_up"] = torch.cat([p[1] for p in parts], 0).contiguous()
        out["Ws_down"] = torch.cat([p[2] for p in parts], 1).contiguous()
        if with_shared_parts:
            out["Ws_parts"] = parts
    else:
        out["Ws_gate"] = out["Ws_up"] = out["Ws_down"] = None
    return out


def equal_logit_router(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """An all-zero router weight: every token sees identical logits for all experts."""
    return torch.zeros((cfg.N, cfg.d_model), dtype=cfg.torch_dtype, device=device)


def small_variant(cfg: MoEConfig, T: int, d_model: int, d_expert: int, d_shared: int,
                  N: Optional[int] = None) -> MoEConfig:
    """The same routing recipe at a reduced size (for parity runs the oracle finishes quickly)."""
    return cfg.replace(name=f"{cfg.name}-small", T=T, d_model=d_model, d_expert=d_expert,
                       d_shared=d_shared if cfg.d_shared > 0 else 0,
                       N=N if N is not None else cfg.N)
