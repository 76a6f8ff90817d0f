"""Shared code of the GPU parity tests: run the layer through the C ABI, run the
oracle on the same inputs, and compare."""
import numpy as np
import torch

import oracle as O
from tests.conftest import ensure_built

ensure_built()

TOL = {"f32": 1e-5, "bf16": 1.5e-2}


def run_layer(spec, inp, staged=False, h_format=None, h_scale_log2=0):
    import routing_shared_expert_gb300 as moe
    cfg = moe.config_from_spec(spec, h_format=h_format, h_scale_log2=h_scale_log2)
    layer = moe.MoELayer(cfg, inp, "cuda")
    if staged:
        layer.forward_staged(inp["x"])
    else:
        layer.forward(inp["x"])
    torch.cuda.synchronize()
    return layer


def host(inp):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}


def check_routing_exact(layer, spec, selection_bias=None):
    """Indices, counts, capacity, offsets, positions and permutation: bit-exact against the
    oracle fed the device's fp32 logits.  Returns the oracle Routing."""
    out = {k: v.cpu() for k, v in layer.out.items()}
    sb = None if selection_bias is None else selection_bias.cpu().numpy()
    rt = O.route(out["logits"].numpy(), spec, selection_bias=sb)
    T, K, N = spec.T, spec.K, spec.N
    np.testing.assert_array_equal(out["topk_idx"].numpy(), rt.topk_idx)
    np.testing.assert_array_equal(out["counts_req"].numpy(), rt.counts_req)
    np.testing.assert_array_equal(out["counts_keep"].numpy(), rt.counts_keep)
    np.testing.assert_array_equal(out["offsets"].numpy(), rt.offsets)
    np.testing.assert_array_equal(out["route_pos"].numpy(), rt.route_pos)
    n_kept = int(rt.offsets[N])
    np.testing.assert_array_equal(out["perm_src"].numpy()[:n_kept], rt.perm_src)
    np.testing.assert_array_equal(out["R_req"].numpy(), rt.R_req)
    np.testing.assert_array_equal(out["R_keep"].numpy(), rt.R_keep)
    ds = out["drop_stats"].numpy()
    assert ds[0] == rt.drops["dropped_routes"]
    assert ds[1] == rt.drops["tokens_lost_any"]
    assert ds[2] == rt.drops["tokens_lost_all"]
    # coefficients: fp32 on the device, fp64 in the oracle
    np.testing.assert_allclose(out["topk_w"].double().numpy(), rt.topk_w, rtol=2e-5, atol=1e-6)
    return rt


def check_logits(layer, spec, inp_host, rows=None):
    z_dev = layer.out["logits"].cpu().double().numpy()
    x = inp_host["x"] if rows is None else inp_host["x"][rows]
    z_ref = O.router_logits(x, inp_host["W_router"], inp_host.get("router_bias"))
    if rows is not None:
        z_dev = z_dev[rows]
    scale = np.sqrt((z_ref ** 2).mean()) + 1e-30
    err = np.abs(z_dev - z_ref).max() / scale
    assert err < 1e-4, f"router logits rel err {err:.3e}"


def oracle_y(spec, inp_host, rt, tokens):
    s = O.shared_coefficient(inp_host["x"][tokens], spec.shared_mode, spec.shared_gain,
                             inp_host.get("shared_gate_w"))
    shared = None
    if spec.d_shared > 0:
        shared = (inp_host["Ws_gate"], inp_host["Ws_up"], inp_host["Ws_down"])
    W = inp_host
    return O.moe_outputs_for_tokens(tokens, inp_host["x"][tokens], rt,
                                    lambda e: (W["W_gate"][e], W["W_up"][e], W["W_down"][e]),
                                    shared, s), s


def rel_err(y, y_ref):
    return float(np.abs(y - y_ref).max() / (np.sqrt((y_ref ** 2).mean()) + 1e-30))


def layer_error(spec, y, y_ref, route_pos):
    """max|y - y_ref| / rms(y_ref), the rms taken over every one of the T*d elements.

    Rows that receive no contribution at all (every route dropped and no shared
    expert) must be exact zeros on both sides; they stay in the rms like every
    other row.
    """
    y = np.asarray(y)
    if spec.d_shared == 0 or spec.shared_mode == "none":
        empty = (np.asarray(route_pos) < 0).all(axis=1)
        assert (y[empty] == 0).all(), "a row with every route dropped must be exactly zero"
        assert (y_ref[empty] == 0).all()
    return rel_err(y, y_ref)


# measured errors of this session, printed beside their bars at the end of the run
ERRORS = []


def record_error(case, err, bar):
    ERRORS.append((case, float(err), float(bar)))


def emulated_y(spec, inp_host, rt, tokens, h_dtype, out_dtype=None):
    """Eq. 80 in float64 with the roundings the device takes: each expert's intermediate
    h = SiLU(x W_g) * (x W_u) rounded to ``h_dtype`` (torch.bfloat16 or torch.float16)
    before the down projection, and, with ``out_dtype``, each expert's output f and the
    shared output g rounded to it before the merge.  Checks the kernels' arithmetic, not
    the method (the oracle does that)."""
    x = torch.as_tensor(inp_host["x"])[torch.as_tensor(tokens)].double()

    def expert(Wg, Wu, Wd, xr):
        a = xr @ Wg.double().T
        b = xr @ Wu.double().T
        h = (a * torch.sigmoid(a) * b).to(h_dtype).double()
        f = h @ Wd.double().T
        if out_dtype is not None:
            f = f.to(out_dtype).double()
        return f.numpy()

    y = np.zeros((len(tokens), spec.d_model))
    idx = rt.topk_idx[tokens]
    kept = rt.route_pos[tokens] >= 0
    r = rt.topk_w[tokens]
    for e in np.unique(idx[kept]):
        rows, slots = np.nonzero((idx == e) & kept)
        y[rows] += r[rows, slots][:, None] * expert(inp_host["W_gate"][e], inp_host["W_up"][e],
                                                    inp_host["W_down"][e], x[rows])
    if spec.d_shared > 0:
        s = O.shared_coefficient(x.numpy(), spec.shared_mode, spec.shared_gain,
                                 inp_host.get("shared_gate_w"))
        y += s[:, None] * expert(inp_host["Ws_gate"], inp_host["Ws_up"], inp_host["Ws_down"], x)
    return y
