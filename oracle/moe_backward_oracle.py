"""Oracle for the backward pass of the routed + shared-expert MoE layer.

TEST INFRASTRUCTURE, like ``moe_oracle``: only the test suite, the smoke check
and the benchmark's CPU legs may import or run it; the library never does.

What it computes ("Section 21: Merging Routed and Shared Expert Activations",
the backward study of Figure 70 (b)-(c): input gradients with the router
coefficients fixed, and with the gradient through the router included; the
routed and shared down-projection weight gradients).  Given the upstream
gradient dy = dL/dy of Eq. 80's output,

    y_t = sum_k r_tk f_{e_tk}(x_t) + s_t g(x_t),
    f_e(x) = W_d^e (SiLU(W_g^e x) * (W_u^e x))            (Eq. 74)

the chain rule gives, per kept route (t, k) with expert e (and the same for the
shared expert with s_t in place of r_tk):

    gf   = r_tk dy_t                      upstream gradient of f
    a    = W_g^e x_t,  b = W_u^e x_t,     h = SiLU(a) * b
    dh   = (W_d^e)^T gf                   dW_d^e += gf h^T
    da   = dh * b * SiLU'(a),  db = dh * SiLU(a)
    dW_g^e += da x_t^T,  dW_u^e += db x_t^T
    dx_t   += (W_g^e)^T da + (W_u^e)^T db

with SiLU(a) = a sigma(a) and SiLU'(a) = sigma(a) (1 + a (1 - sigma(a))).

With the router differentiable, the coefficients carry gradient too:
dr_tk = dy_t . f_{e_tk}(x_t) and ds_t = dy_t . g(x_t); r = alpha w(q(z)) is
differentiated through the selected-weight rule of Table 52 and the score map
(softmax over all N, or sigmoid), back to the logits z = W_r x (+ bias), so
dW_r += dz x^T and dx += W_r^T dz; a learned shared gate s = sigma(w_s . x)
(Eq. 77) adds dw_s += ds s (1 - s) x and dx += ds s (1 - s) w_s.  The selection
itself is piecewise constant in z: the selected set and the kept routes are held
fixed, as the forward pass decided them.

Readings: a dropped route contributes nothing and carries no gradient; the
logit bias and the selection-only bias are inputs, not parameters (no gradient
is formed for them); the Eq. 35 selection bias changes only which experts are
selected, so it enters the backward pass only through the fixed selection.

Everything is float64.  Pinned in tests/test_oracle_backward_pins.py by central
finite differences of the forward oracle and by the Eq. 81 dense reduction.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from .moe_oracle import (F64, f64, moe_forward, route, router_logits, selection_keys,
                         shared_coefficient, sigmoid, silu, softmax_all)


def dsilu(a) -> np.ndarray:
    """d SiLU(a) / da = sigma(a) (1 + a (1 - sigma(a)))."""
    a = f64(a)
    s = sigmoid(a)
    return s * (1.0 + a * (1.0 - s))


def swiglu_backward(x, W_gate, W_up, W_down, gf):
    """Backward of f = W_d (SiLU(W_g x) * (W_u x)) for rows x [n, d] and upstream
    gradients gf [n, d] (Eq. 74).  Returns (dx [n, d], dW_gate, dW_up, dW_down)."""
    x, Wg, Wu, Wd, gf = f64(x), f64(W_gate), f64(W_up), f64(W_down), f64(gf)
    a = x @ Wg.T
    b = x @ Wu.T
    h = silu(a) * b
    dh = gf @ Wd                        # [n, d_r]
    dWd = gf.T @ h                      # [d, d_r]
    da = dh * b * dsilu(a)
    db = dh * silu(a)
    dWg = da.T @ x                      # [d_r, d]
    dWu = db.T @ x
    dx = da @ Wg + db @ Wu
    return dx, dWg, dWu, dWd


def selected_weights_backward(z, idx, score: str, norm: str, dw, p: float = 2.0) -> np.ndarray:
    """dL/dz [T, N] from dL/dw [T, K] for the selected-weight rules of Table 52
    (see ``moe_oracle.selected_weights``), the selection idx held fixed."""
    z = f64(z)
    dw = f64(dw)
    T, N = z.shape
    idx = np.asarray(idx)
    dz = np.zeros((T, N), F64)
    rows = np.arange(T)[:, None]
    if norm == "softmax_selected":
        zS = np.take_along_axis(z, idx, axis=1)
        w = np.exp(zS - zS.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        # dz_S = w * (dw - sum_k w_k dw_k)
        g = w * (dw - (w * dw).sum(axis=1, keepdims=True))
        np.add.at(dz, (np.broadcast_to(rows, idx.shape), idx), g)
        return dz
    q = softmax_all(z) if score == "softmax" else sigmoid(z)
    qS = np.take_along_axis(q, idx, axis=1)
    # dL/dq_S through the normalisation
    if norm == "none":
        dqS = dw
    elif norm == "l1":
        S = qS.sum(axis=1, keepdims=True)
        w = qS / S
        dqS = (dw - (w * dw).sum(axis=1, keepdims=True)) / S
    elif norm == "lp":
        n = np.power(np.power(qS, p).sum(axis=1, keepdims=True), 1.0 / p)
        w = qS / n
        # w_k = q_k / n,  dn/dq_m = (q_m / n)^(p-1)
        dqS = dw / n - (w * dw).sum(axis=1, keepdims=True) * np.power(w, p - 1.0) / n
    else:
        raise ValueError(norm)
    dq = np.zeros((T, N), F64)
    np.add.at(dq, (np.broadcast_to(rows, idx.shape), idx), dqS)
    if score == "softmax":
        # dz_j = q_j (dq_j - sum_i q_i dq_i)
        dz = q * (dq - (q * dq).sum(axis=1, keepdims=True))
    else:
        dz = dq * q * (1.0 - q)
    return dz


def moe_backward(cfg, inputs: dict, dy, router_grad: bool = False,
                 logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Gradients of the layer of ``moe_oracle.moe_forward`` for upstream gradient
    dy [T, d].  ``router_grad`` False holds the coefficients r and s fixed (the
    expert-path Jacobian); True adds the gradient through them.  Returns a dict
    with dx, dW_gate, dW_up, dW_down [N, ...], and for a shared expert dWs_gate,
    dWs_up, dWs_down; with ``router_grad`` also dW_router and, for a learned
    shared gate, dshared_gate_w."""
    x = f64(inputs["x"])
    dy = f64(dy)
    T, d = x.shape
    z = router_logits(inputs["x"], inputs["W_router"], inputs.get("router_bias")) if logits is None \
        else f64(logits)
    rt = route(z, cfg, selection_bias=inputs.get("selection_bias"))
    s = shared_coefficient(inputs["x"], cfg.shared_mode, cfg.shared_gain, inputs.get("shared_gate_w"))
    Wg, Wu, Wd = inputs["W_gate"], inputs["W_up"], inputs["W_down"]
    N, K = cfg.N, cfg.K
    out = {"dx": np.zeros((T, d), F64)}
    dWg = np.zeros((N,) + tuple(Wg.shape[1:]), F64)
    dWu = np.zeros_like(dWg)
    dWd = np.zeros((N,) + tuple(Wd.shape[1:]), F64)
    dr = np.zeros((T, K), F64)
    kept = rt.route_pos >= 0
    for e in np.unique(rt.topk_idx[kept]):
        e = int(e)
        toks, slots = np.nonzero((rt.topk_idx == e) & kept)
        gf = rt.topk_w[toks, slots][:, None] * dy[toks]
        dxe, g1, g2, g3 = swiglu_backward(x[toks], Wg[e], Wu[e], Wd[e], gf)
        np.add.at(out["dx"], toks, dxe)
        dWg[e] += g1
        dWu[e] += g2
        dWd[e] += g3
        if router_grad:
            from .moe_oracle import swiglu
            f = swiglu(x[toks], Wg[e], Wu[e], Wd[e])
            dr[toks, slots] = (dy[toks] * f).sum(axis=1)
    out.update(dW_gate=dWg, dW_up=dWu, dW_down=dWd)
    shared = cfg.d_shared > 0 and cfg.shared_mode != "none"
    if shared:
        gs = f64(s)[:, None] * dy
        dxs, g1, g2, g3 = swiglu_backward(x, inputs["Ws_gate"], inputs["Ws_up"], inputs["Ws_down"], gs)
        out["dx"] += dxs
        out.update(dWs_gate=g1, dWs_up=g2, dWs_down=g3)
    if router_grad:
        dw = cfg.alpha * dr                     # r = alpha w
        dz = selected_weights_backward(z, rt.topk_idx, cfg.score, cfg.norm, dw,
                                       getattr(cfg, "norm_p", 2.0))
        Wr = f64(inputs["W_router"])
        out["dW_router"] = dz.T @ x
        out["dx"] += dz @ Wr
        if shared and cfg.shared_mode == "gate":
            from .moe_oracle import swiglu
            g = swiglu(x, inputs["Ws_gate"], inputs["Ws_up"], inputs["Ws_down"])
            ds = (dy * g).sum(axis=1)
            du = ds * f64(s) * (1.0 - f64(s))
            w_s = f64(inputs["shared_gate_w"])
            out["dshared_gate_w"] = du @ x
            out["dx"] += du[:, None] * w_s[None, :]
    return out
