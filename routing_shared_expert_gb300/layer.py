"""A convenience holder for one MoE layer on the device: config, weights, workspace, outputs.

Marshalling only.  ``forward`` is one ``moe_layer_forward`` call; ``forward_staged``
runs the same five entry points one by one (optionally recording CUDA events
between them on the launching stream, which is how per-kernel times are taken).
With the fp16 intermediate (the default for bf16 layers) the down projections are
packed once, at construction, by ``moe_pack_weights``; the backward pass reads the
bf16 tensors as given.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import _native as nat


def config_from_spec(spec, T: Optional[int] = None, h_format: Optional[str] = None,
                     h_scale_log2: int = 0) -> nat.moe_config:
    """A ``moe_config`` from any object with the layer's fields (T, d_model, N, K, ...).

    ``h_format`` defaults to the spec's own field if it has one, else "f16" (the fp16
    intermediate with packed down projections) for bf16 layers."""
    if h_format is None:
        h_format = getattr(spec, "h_format", None) or ("f16" if spec.dtype == "bf16" else "bf16")
    return nat.make_config(
        T=spec.T if T is None else T, d_model=spec.d_model, N=spec.N, K=spec.K,
        d_expert=spec.d_expert, d_shared=spec.d_shared, dtype=spec.dtype, score=spec.score,
        norm=spec.norm, alpha=spec.alpha, shared_mode=spec.shared_mode,
        shared_gain=spec.shared_gain, cap_policy=spec.cap_policy,
        capacity_factor=spec.capacity_factor, num_ranks=spec.num_ranks,
        rho=[i % spec.num_ranks for i in range(spec.N)], norm_p=getattr(spec, "norm_p", 2.0),
        h_format=h_format, h_scale_log2=h_scale_log2)


STAGES = ("route", "permute", "grouped_swiglu", "shared_mlp", "combine")


class MoELayer:
    def __init__(self, cfg: nat.moe_config, weights: Dict[str, Optional[torch.Tensor]],
                 device="cuda", staged_buffers: bool = True):
        self.cfg = cfg
        self.device = torch.device(device)
        self.weights = weights
        self.h_f16 = cfg.dtype == nat.DTYPES["bf16"] and cfg.h_format == nat.H_FORMATS["f16"]
        # the down projections the forward reads: packed fp16 buffers for the fp16 intermediate
        self.down = {"W_down": weights["W_down"], "Ws_down": weights.get("Ws_down")}
        if self.h_f16:
            self.down = {k: (nat.pack_weights(v) if v is not None else None)
                         for k, v in self.down.items()}
        self.w = self._weights(self.down)
        self.ws = nat.alloc_workspace(cfg, device)
        T, d, N, K, M = cfg.T, cfg.d_model, cfg.N, cfg.K, cfg.num_ranks
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.out = {
            "y": torch.empty((T, d), **f32),
            "topk_idx": torch.empty((T, K), **i32),
            "topk_w": torch.empty((T, K), **f32),
            "shared_coef": torch.empty((T,), **f32),
            "logits": torch.empty((T, N), **f32),
            "counts_req": torch.empty((N,), **i32),
            "counts_keep": torch.empty((N,), **i32),
            "offsets": torch.empty((N + 1,), **i32),
            "route_pos": torch.empty((T, K), **i32),
            "perm_src": torch.empty((T * K,), **i32),
            "R_req": torch.empty((M,), **i32),
            "R_keep": torch.empty((M,), **i32),
            "drop_stats": torch.empty((4,), **i32),
        }
        self.outputs = nat.make_outputs(**self.out)
        self.staged = None
        if staged_buffers:
            dt = torch.float32 if cfg.dtype == nat.DTYPES["f32"] else torch.bfloat16
            # expert outputs: fp16 (holding f 2^-h_scale_log2) under the fp16 intermediate
            ft = torch.float16 if self.h_f16 else torch.float32
            self.staged = {
                "x_perm": torch.empty((T * K, d), dtype=dt, device=device),
                "f": torch.empty((T * K, d), dtype=ft, device=device),
                "g": torch.empty((T, d), dtype=ft, device=device) if cfg.d_shared > 0 else None,
            }

    def _weights(self, down):
        w = self.weights
        return nat.make_weights(w["W_router"], w.get("router_bias"), w.get("shared_gate_w"),
                                w["W_gate"], w["W_up"], down["W_down"], w.get("Ws_gate"),
                                w.get("Ws_up"), down["Ws_down"], w.get("selection_bias"))

    def forward(self, x: torch.Tensor, stream=None, logits: bool = True) -> torch.Tensor:
        outs = self.outputs if logits else self._no_logits()
        nat.moe_layer_forward(self.cfg, self.w, x, outs, self.ws, stream)
        return self.out["y"]

    def forward_profiled(self, x: torch.Tensor, events, stream=None, logits: bool = False):
        """forward() with 5 events recorded inside the call (see moe_layer_forward_profiled)."""
        outs = self.outputs if logits else self._no_logits()
        nat.moe_layer_forward_profiled(self.cfg, self.w, x, outs, self.ws, events, stream)
        return self.out["y"]

    def _no_logits(self):
        if not hasattr(self, "_outputs_nolog"):
            d = {k: v for k, v in self.out.items() if k != "logits"}
            self._outputs_nolog = nat.make_outputs(**d)
        return self._outputs_nolog

    def forward_staged(self, x: torch.Tensor, events=None, stream=None) -> torch.Tensor:
        """The five entry points in order; ``events`` (len 6) are recorded around them."""
        c, o, s, w = self.cfg, self.out, self.staged, self.weights
        st = stream if stream is not None else torch.cuda.current_stream()

        def rec(i):
            if events is not None:
                events[i].record(st)

        rec(0)
        nat.moe_route(c, x, w["W_router"], w.get("router_bias"), w.get("selection_bias"),
                      w.get("shared_gate_w"), o["topk_idx"], o["topk_w"], o["shared_coef"],
                      o["logits"], self.ws, st)
        rec(1)
        nat.moe_permute(c, x, o["topk_idx"], o["counts_req"], o["counts_keep"], o["offsets"],
                        o["route_pos"], o["perm_src"], s["x_perm"], o["R_req"], o["R_keep"],
                        o["drop_stats"], self.ws, st)
        rec(2)
        nat.moe_grouped_swiglu(c, s["x_perm"], o["offsets"], None, w["W_gate"], w["W_up"],
                               self.down["W_down"], s["f"], self.ws, st)
        rec(3)
        if c.d_shared > 0:
            nat.moe_shared_mlp(c, x, w["Ws_gate"], w["Ws_up"], self.down["Ws_down"], s["g"],
                               self.ws, st)
        rec(4)
        nat.moe_combine(c, s["f"], o["route_pos"], o["topk_w"], s["g"],
                        o["shared_coef"] if c.d_shared > 0 else None, o["y"], st)
        rec(5)
        return o["y"]

    def backward(self, x: torch.Tensor, dy: torch.Tensor, stream=None,
                 router_grad: bool = False) -> Dict[str, torch.Tensor]:
        """Gradients for upstream gradient dy [T][d] fp32, using the routing of the last
        forward call (which must have written the logits when ``router_grad``); returns dx
        and the weight gradients (fp32).  ``router_grad`` adds the gradient through the
        router coefficients (dW_router, and dshared_gate_w for a learned shared gate)."""
        if not hasattr(self, "cfg_bwd"):
            # the backward reads the bf16 down projections: a configuration that says so
            self.cfg_bwd = nat.copy_config(self.cfg, h_format=nat.H_FORMATS["bf16"])
            self.w_bwd = self._weights({"W_down": self.weights["W_down"],
                                        "Ws_down": self.weights.get("Ws_down")})
        c = self.cfg_bwd
        if getattr(self, "_bwd_router", None) != router_grad:
            self.bwd_ws = None
            self._bwd_router = router_grad
        if getattr(self, "bwd_ws", None) is None:
            n = nat.moe_backward_workspace_size(c)
            self.bwd_ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
            nat.moe_workspace_init(self.bwd_ws, stream)
            f32 = dict(dtype=torch.float32, device=self.device)
            T, d, N, dr, ds = c.T, c.d_model, c.N, c.d_expert, c.d_shared
            self.grads = {"dx": torch.empty((T, d), **f32),
                          "dW_gate": torch.empty((N, dr, d), **f32),
                          "dW_up": torch.empty((N, dr, d), **f32),
                          "dW_down": torch.empty((N, d, dr), **f32)}
            if ds > 0:
                self.grads.update(dWs_gate=torch.empty((ds, d), **f32), dWs_up=torch.empty((ds, d), **f32),
                                  dWs_down=torch.empty((d, ds), **f32))
            if router_grad:
                self.grads["dW_router"] = torch.empty((N, d), **f32)
                if c.shared_mode == nat.SHARED_MODES["gate"]:
                    self.grads["dshared_gate_w"] = torch.empty((d,), **f32)
            self.grads_c = nat.make_grads(**self.grads)
        nat.moe_layer_backward(c, self.w_bwd, x, self.outputs, dy, self.grads_c, self.bwd_ws, stream)
        return self.grads

    def backward_status(self) -> int:
        return nat.moe_read_status(self.bwd_ws)

    def status(self) -> int:
        return nat.moe_read_status(self.ws)
