"""Backward pass of the layer with the router coefficients fixed, on a GB300, against the
float64 oracle (oracle.moe_backward, pinned by finite differences): dx and every weight
gradient within the bf16 bar, with the oracle run on the device's own routing."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_helpers import check_routing_exact, host, run_layer
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

# Bars of the backward against the float64 oracle.  Every GEMM product has its two
# operands rounded to bf16 once (unit roundoff u = 2^-8) among gf = r dy, h, da, db, so
# each term of a gradient element carries a relative error up to ~2u = 7.8e-3.  Over a
# tensor the errors are independent: the rms of the error stays near 0.8 u = 3e-3 of the
# rms of the tensor, and the bar on it is the forward's bf16 bar, 1.5e-2.  The largest
# single error is bounded by ~2u times the largest element, and a weight-gradient element
# of an expert with few rows (DeepSeek-V3 shape: ~20) sums few products and reaches ~10x
# the tensor's rms: the bar on max|error| / rms is 1e-1.  The kernels' own arithmetic is
# checked against the same rounding emulated in float64 (rms 1e-3; max 6e-2, since the
# emulation rounds float64 values where the kernels round fp32 ones and a few operands
# fall on the other side of a rounding boundary, one bf16 ulp on a large element).
BWD_RMS_TOL = 1.5e-2
BWD_MAX_TOL = 1e-1

C = CONFIGS
SHAPES = {
    # d, d_r, d_s multiples of 128; T ragged against the 64-row padding and 128-row tiles
    "olmo_s": C["olmo"].replace(T=1000, d_model=512, d_expert=384, d_shared=256),
    "dsv3_s": C["dsv3"].replace(T=600, d_model=512, d_expert=128, d_shared=128),
    "qwen2_s": C["qwen2"].replace(T=777, d_model=256, d_expert=256, d_shared=384),
    "mixtral_cap": C["mixtral"].replace(T=700, d_model=1024, d_expert=512, capacity_factor=0.6),
    "olmo_k1": C["olmo"].replace(T=300, d_model=256, d_expert=128, d_shared=128, K=1, alpha=1.0),
}


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _emulated(spec, hin, dy, fwd):
    """The same backward with the kernels' rounding: dy, r h, da, db rounded to bf16,
    everything else float64 (a diagnostic reference for the kernel arithmetic)."""
    x = O.f64(hin["x"])
    T, d = x.shape
    idx = fwd["topk_idx"]
    w = fwd["topk_w"]
    pos = fwd["route_pos"]
    out = {"dx": np.zeros((T, d))}
    N = spec.N
    dWg = np.zeros((N,) + tuple(hin["W_gate"].shape[1:]))
    dWu = np.zeros_like(dWg)
    dWd = np.zeros((N,) + tuple(hin["W_down"].shape[1:]))

    def fam(xr, dyr, sc, Wg, Wu, Wd):
        # the kernels: dh = c (dy_bf16 W_d), dW_d = dy_bf16^T bf16(c h)
        a = xr @ Wg.T
        b = xr @ Wu.T
        hf = O.silu(a) * b
        dh = sc[:, None] * (dyr @ Wd)
        da = _bf16(dh * b * O.dsilu(a))
        db = _bf16(dh * O.silu(a))
        return da @ Wg + db @ Wu, da.T @ xr, db.T @ xr, dyr.T @ _bf16(sc[:, None] * hf)

    dyb = _bf16(dy)
    for e in range(N):
        toks, slots = np.nonzero((idx == e) & (pos >= 0))
        if len(toks) == 0:
            continue
        dxe, g1, g2, g3 = fam(x[toks], dyb[toks], w[toks, slots], O.f64(hin["W_gate"][e]),
                              O.f64(hin["W_up"][e]), O.f64(hin["W_down"][e]))
        np.add.at(out["dx"], toks, dxe)
        dWg[e], dWu[e], dWd[e] = g1, g2, g3
    out.update(dW_gate=dWg, dW_up=dWu, dW_down=dWd)
    if spec.d_shared:
        dxs, g1, g2, g3 = fam(x, dyb, fwd["shared_coef"], O.f64(hin["Ws_gate"]), O.f64(hin["Ws_up"]),
                              O.f64(hin["Ws_down"]))
        out["dx"] += dxs
        out.update(dWs_gate=g1, dWs_up=g2, dWs_down=g3)
    return out


def _rms_rel(a, b):
    """rms(a - b) / rms(b): the emulated reference rounds float64 values where the kernels
    round fp32 ones, so a few elements land on the other side of a bf16 rounding boundary;
    those one-ulp flips stay far below any real defect in this measure."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.sqrt(((a - b) ** 2).mean() / max((b ** 2).mean(), 1e-300)))


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    rms = np.sqrt((b ** 2).mean())
    return float(np.abs(a - b).max() / rms) if rms > 0 else float(np.abs(a - b).max())


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_router_fixed(name):
    spec = SHAPES[name]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp)
    assert layer.status() == 0
    rt = check_routing_exact(layer, spec)
    g = torch.Generator(device="cpu").manual_seed(7)
    dy = torch.randn((spec.T, spec.d_model), generator=g).to("cuda")
    grads = layer.backward(inp["x"], dy)
    torch.cuda.synchronize()
    assert layer.backward_status() == 0
    hin = host(inp)
    ref = O.moe_backward(spec, hin, dy.cpu().numpy(), router_grad=False,
                         logits=layer.out["logits"].cpu().numpy())
    keys = ["dx", "dW_gate", "dW_up", "dW_down"] + (["dWs_gate", "dWs_up", "dWs_down"] if spec.d_shared else [])
    got = {k: grads[k].cpu().numpy() for k in keys}
    # the kernels' arithmetic: against the same rounding of the intermediates, fp32
    # accumulation order is all that differs
    fwd = {k: v.cpu().numpy().astype(np.float64) if v.dtype.is_floating_point else v.cpu().numpy()
           for k, v in layer.out.items()}
    emu = _emulated(spec, hin, dy.cpu().numpy().astype(np.float64), fwd)
    for k in keys:
        er, em = _rms_rel(got[k], emu[k]), _rel(got[k], emu[k])
        assert er <= 1e-3 and em <= 6e-2, f"{name} {k}: vs emulated rounding rms {er:.3e} max {em:.3e}"
    # against the float64 definition
    for k in keys:
        er, em = _rms_rel(got[k], ref[k]), _rel(got[k], ref[k])
        assert er <= BWD_RMS_TOL and em <= BWD_MAX_TOL, f"{name} {k}: rms {er:.3e} max {em:.3e}"
    if spec.cap_policy != "none":
        assert rt.drops["dropped_routes"] > 0


def test_backward_twice_same_result():
    spec = SHAPES["olmo_s"]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp)
    dy = torch.randn((spec.T, spec.d_model), device="cuda")
    a = {k: v.clone() for k, v in layer.backward(inp["x"], dy).items()}
    b = layer.backward(inp["x"], dy)
    torch.cuda.synchronize()
    assert layer.backward_status() == 0
    for k in a:
        assert torch.equal(a[k], b[k]), k


ROUTER_SHAPES = {
    # the selected-weight rules of Table 52 and the learned shared gate (Eq. 77)
    "olmo_l1": SHAPES["olmo_s"],                                                    # softmax, L1, alpha = K
    "qwen2_none_gate": SHAPES["qwen2_s"],                                           # softmax, none, sigmoid gate
    "dsv3_sigmoid_l1": SHAPES["dsv3_s"],                                            # sigmoid, L1, alpha = 2.5
    "mixtral_selected": SHAPES["mixtral_cap"],                                      # softmax over selected, drops
    "olmo_lp3": SHAPES["olmo_k1"].replace(K=2, norm="lp", norm_p=3.0, alpha=2.0),   # L_p
}


@pytest.mark.parametrize("name", list(ROUTER_SHAPES))
def test_backward_through_router(name):
    spec = ROUTER_SHAPES[name]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp)
    assert layer.status() == 0
    check_routing_exact(layer, spec)
    g = torch.Generator(device="cpu").manual_seed(11)
    dy = torch.randn((spec.T, spec.d_model), generator=g).to("cuda")
    grads = layer.backward(inp["x"], dy, router_grad=True)
    torch.cuda.synchronize()
    assert layer.backward_status() == 0
    hin = host(inp)
    ref = O.moe_backward(spec, hin, dy.cpu().numpy(), router_grad=True,
                         logits=layer.out["logits"].cpu().numpy())
    keys = ["dx", "dW_router", "dW_down"] + (["dshared_gate_w"] if spec.shared_mode == "gate" else [])
    for k in keys:
        got = grads[k].cpu().numpy()
        er, em = _rms_rel(got, ref[k]), _rel(got, ref[k])
        assert er <= BWD_RMS_TOL and em <= BWD_MAX_TOL, f"{name} {k}: rms {er:.3e} max {em:.3e}"

