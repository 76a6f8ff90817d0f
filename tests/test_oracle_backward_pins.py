"""Pins of the backward oracle (CPU only): central finite differences of the forward
oracle, and the Eq. 81 dense reduction.

The backward study of "Section 21: Merging Routed and Shared Expert Activations"
(Figure 70 (b)-(c)) reports input gradients with the router coefficients fixed and
with the gradient through the router, and the routed / shared down-projection weight
gradients.  Finite differences of the forward pass pin every one of those derivatives
independently of the analytic chain rule the oracle writes out.
"""
import itertools

import numpy as np
import pytest

import oracle as O


class Cfg:
    def __init__(self, **kw):
        self.__dict__.update(dict(score="softmax", norm="l1", alpha=2.0, cap_policy="none",
                                  capacity_factor=1.0, num_ranks=1, shared_mode="const",
                                  shared_gain=1.0, norm_p=2.0))
        self.__dict__.update(kw)


def _layer(seed, T=5, d=6, N=4, K=2, dr=3, ds=2, gate=False):
    rng = np.random.default_rng(seed)
    inp = {
        "x": rng.normal(size=(T, d)),
        "W_router": rng.normal(size=(N, d)) * 0.7,
        "W_gate": rng.normal(size=(N, dr, d)) * 0.5,
        "W_up": rng.normal(size=(N, dr, d)) * 0.5,
        "W_down": rng.normal(size=(N, d, dr)) * 0.5,
    }
    if ds:
        inp.update(Ws_gate=rng.normal(size=(ds, d)) * 0.5, Ws_up=rng.normal(size=(ds, d)) * 0.5,
                   Ws_down=rng.normal(size=(d, ds)) * 0.5)
    if gate:
        inp["shared_gate_w"] = rng.normal(size=(d,)) * 0.5
    dy = rng.normal(size=(T, d))
    return inp, dy


def _loss(cfg, inp, dy, idx, route_pos, router_grad):
    """L = sum(dy * y) with the selection (and the kept routes) held at idx / route_pos;
    coefficients recomputed from the inputs when router_grad, else taken from base."""
    x = inp["x"]
    z = O.router_logits(x, inp["W_router"])
    w = O.selected_weights(z, idx, cfg.score, cfg.norm, cfg.norm_p)
    r = cfg.alpha * w
    s = O.shared_coefficient(x, cfg.shared_mode, cfg.shared_gain, inp.get("shared_gate_w"))
    if not router_grad:
        r, s = cfg._r, cfg._s
    y = np.zeros_like(x)
    for t in range(x.shape[0]):
        for k in range(cfg.K):
            if route_pos[t, k] < 0:
                continue
            e = idx[t, k]
            y[t] += r[t, k] * O.swiglu(x[t:t + 1], inp["W_gate"][e], inp["W_up"][e], inp["W_down"][e])[0]
    if cfg.d_shared:
        y += s[:, None] * O.swiglu(x, inp["Ws_gate"], inp["Ws_up"], inp["Ws_down"])
    return float((dy * y).sum())


def _fd_check(cfg, inp, dy, router_grad, names, h=1e-6, rtol=1e-6):
    cfg.T, cfg.N = inp["x"].shape[0], inp["W_router"].shape[0]
    z = O.router_logits(inp["x"], inp["W_router"])
    rt = O.route(z, cfg)
    cfg._r = rt.topk_w
    cfg._s = O.shared_coefficient(inp["x"], cfg.shared_mode, cfg.shared_gain, inp.get("shared_gate_w"))
    g = O.moe_backward(cfg, inp, dy, router_grad=router_grad)
    key = {"x": "dx", "W_gate": "dW_gate", "W_up": "dW_up", "W_down": "dW_down", "Ws_gate": "dWs_gate",
           "Ws_up": "dWs_up", "Ws_down": "dWs_down", "W_router": "dW_router",
           "shared_gate_w": "dshared_gate_w"}
    for name in names:
        base = inp[name]
        num = np.zeros_like(base)
        for i in np.ndindex(base.shape):
            old = base[i]
            base[i] = old + h
            lp = _loss(cfg, inp, dy, rt.topk_idx, rt.route_pos, router_grad)
            base[i] = old - h
            lm = _loss(cfg, inp, dy, rt.topk_idx, rt.route_pos, router_grad)
            base[i] = old
            num[i] = (lp - lm) / (2 * h)
        ana = g[key[name]]
        scale = max(np.abs(num).max(), 1e-12)
        assert np.abs(ana - num).max() <= rtol * scale + 1e-9, (name, np.abs(ana - num).max(), scale)
    return g


def test_router_fixed_gradients_match_finite_differences():
    inp, dy = _layer(1)
    cfg = Cfg(K=2, d_shared=2)
    _fd_check(cfg, inp, dy, False, ["x", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"])


@pytest.mark.parametrize("score,norm", [("softmax", "l1"), ("softmax", "none"), ("softmax", "softmax_selected"),
                                        ("sigmoid", "l1"), ("softmax", "lp"), ("sigmoid", "lp")])
def test_router_gradients_match_finite_differences(score, norm):
    inp, dy = _layer(2)
    cfg = Cfg(K=2, d_shared=2, score=score, norm=norm, alpha=2.5, norm_p=3.0)
    _fd_check(cfg, inp, dy, True, ["x", "W_router", "W_down"])


def test_learned_shared_gate_gradient_matches_finite_differences():
    inp, dy = _layer(3, gate=True)
    cfg = Cfg(K=2, d_shared=2, norm="none", alpha=1.0, shared_mode="gate")
    _fd_check(cfg, inp, dy, True, ["x", "shared_gate_w", "W_router", "Ws_down"])
    # with the router fixed the gate is a constant: no gate gradient is formed
    g = O.moe_backward(cfg, inp, dy, router_grad=False)
    assert "dshared_gate_w" not in g


def test_dropped_routes_carry_no_gradient():
    inp, dy = _layer(4, T=8, N=4, K=2)
    cfg = Cfg(K=2, d_shared=2, cap_policy="per_expert", capacity_factor=0.5)
    cfg.T, cfg.N = 8, 4
    rt = O.route(O.router_logits(inp["x"], inp["W_router"]), cfg)
    assert (rt.route_pos < 0).any()
    _fd_check(cfg, inp, dy, False, ["x", "W_down"])
    _fd_check(cfg, inp, dy, True, ["x", "W_router"])


def test_eq81_dense_reduction_backward():
    """Equal logits and the Olmo rule (K experts, r = 1 each, s = 1): the layer is one dense
    SwiGLU whose gate/up rows are the selected experts' and the shared expert's, and whose
    down columns are theirs too (Eq. 81-82); its input and weight gradients are those of that
    dense MLP."""
    rng = np.random.default_rng(5)
    T, d, N, K, dr, ds = 7, 6, 4, 2, 3, 2
    inp = {"x": rng.normal(size=(T, d)), "W_router": np.zeros((N, d)),
           "W_gate": rng.normal(size=(N, dr, d)), "W_up": rng.normal(size=(N, dr, d)),
           "W_down": rng.normal(size=(N, d, dr)), "Ws_gate": rng.normal(size=(ds, d)),
           "Ws_up": rng.normal(size=(ds, d)), "Ws_down": rng.normal(size=(d, ds))}
    dy = rng.normal(size=(T, d))
    cfg = Cfg(K=K, N=N, T=T, d_shared=ds, alpha=float(K))
    g = O.moe_backward(cfg, inp, dy, router_grad=False)
    Wg = np.concatenate([inp["W_gate"][0], inp["W_gate"][1], inp["Ws_gate"]])
    Wu = np.concatenate([inp["W_up"][0], inp["W_up"][1], inp["Ws_up"]])
    Wd = np.concatenate([inp["W_down"][0], inp["W_down"][1], inp["Ws_down"]], axis=1)
    dx, dWg, dWu, dWd = O.swiglu_backward(inp["x"], Wg, Wu, Wd, dy)
    np.testing.assert_allclose(g["dx"], dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW_down"][0], dWd[:, :dr], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dWs_down"], dWd[:, 2 * dr:], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW_gate"][1], dWg[dr:2 * dr], rtol=1e-12, atol=1e-12)
    assert np.abs(g["dW_gate"][2:]).max() == 0.0   # experts 2, 3 never selected


def test_dsilu_closed_form():
    # SiLU'(0) = 1/2; SiLU'(a) -> 1 for large a, -> 0 for very negative a
    assert O.dsilu(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(O.dsilu(np.array([40.0])), [1.0], rtol=1e-12)
    np.testing.assert_allclose(O.dsilu(np.array([-40.0])), [0.0], atol=1e-15)
    a = np.linspace(-3, 3, 13)
    h = 1e-6
    np.testing.assert_allclose(O.dsilu(a), (O.silu(a + h) - O.silu(a - h)) / (2 * h), rtol=1e-8)
