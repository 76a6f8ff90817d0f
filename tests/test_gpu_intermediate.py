"""The intermediate format of the bf16 expert GEMMs, on a GB300 (through the C ABI).

The down projection f = h W_d (Section 20, Eq. 74) multiplies the intermediate h by
the down weights on the tensor cores, both in one 16-bit type.  MOE_H_F16 (the default
of the layer holder) keeps h in fp16, reads W_d from a buffer moe_pack_weights wrote
once (fp16 W 2^k) and hands the expert outputs f and g to the combine in fp16;
MOE_H_BF16 keeps h in bf16, reads W_d as given and keeps f and g in fp32.

- The packing is exact for bf16 weights: packed * 2^-k equals W bit for bit, for
  ordinary, tiny, huge and ragged tensors; a non-finite weight is flagged.
- Each format's kernels compute what their rounding says: y against Eq. 80 in float64
  with h rounded to that format, by the rms of the difference (a single h element that
  the device's fp32 rounds across a rounding boundary, where the float64 emulation does
  not, moves one output by up to about an ulp of h times a weight, so the largest
  difference says little); the bf16 layer's error against the oracle is recorded beside
  the spec bar.
- An h past the fp16 range is reported as MOE_ERR_RANGE, and h_scale_log2 brings it back
  (then parity holds); a down pointer that is not a packed buffer of the layer's size is
  reported as MOE_ERR_BAD_PACK.
"""
import math

import numpy as np
import pytest
import torch

import routing_shared_expert_gb300 as moe
from tests.gpu_helpers import (TOL, check_routing_exact, emulated_y, host, layer_error, oracle_y,
                               record_error, rel_err, run_layer)
from tests.test_gpu_parity import SMALL
from workloads import make_inputs

pytestmark = pytest.mark.gpu

RANGE = -8
BAD_PACK = -9
BF16_CASES = [n for n, s in SMALL.items() if s.dtype == "bf16"]


def _header(packed):
    h = packed[:256].cpu()
    return {"magic": int(h[0:4].view(torch.int32)[0]) & 0xFFFFFFFF,
            "absmax": float(h[4:8].view(torch.float32)[0]),
            "k": int(h[8:12].view(torch.int32)[0]),
            "inv_scale": float(h[12:16].view(torch.float32)[0]),
            "elements": int(h[16:24].view(torch.int64)[0]),
            "flags": int(h[24:28].view(torch.int32)[0])}


def _values(packed, n):
    return packed[256:256 + 2 * n].view(torch.float16)


@pytest.mark.parametrize("scale,n", [(1.0, None), (2.0 ** -100, None), (2.0 ** 100, None),
                                     (1.0, 1001), (1.0, 7)])
def test_pack_is_exact(scale, n):
    W = make_inputs(SMALL["olmo_s"], "cuda")["W_down"]
    W = (W.float() * scale).to(torch.bfloat16)
    if n is not None:
        W = W.reshape(-1)[:n].contiguous()
    packed = moe.pack_weights(W)
    torch.cuda.synchronize()
    hd = _header(packed)
    assert hd["magic"] == 0x3631444D and hd["flags"] == 0 and hd["elements"] == W.numel()
    amax = float(W.float().abs().max())
    assert hd["absmax"] == amax
    e = math.frexp(amax)[1]                     # amax in [2^(e-1), 2^e)
    assert hd["k"] == 15 - e and hd["inv_scale"] == 2.0 ** -hd["k"]
    v = _values(packed, W.numel()).double()
    assert 2.0 ** 14 <= float(v.abs().max()) < 2.0 ** 15
    back = v * 2.0 ** -hd["k"]
    Wd = W.double().reshape(-1)
    # exact wherever W 2^k is at least 2^-17 (8 significant bits fit fp16's subnormal
    # spacing 2^-24), which is every weight above max |W| 2^-31; below, within half of it
    big = Wd.abs() * 2.0 ** hd["k"] >= 2.0 ** -17
    assert torch.equal(back[big], Wd[big])
    assert float((back - Wd).abs().max()) <= 2.0 ** -25 * 2.0 ** -hd["k"]


def test_pack_of_zeros_and_flags_of_non_finite_weights():
    Z = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    p = moe.pack_weights(Z)
    torch.cuda.synchronize()
    hd = _header(p)
    assert hd["k"] == 0 and hd["flags"] == 0 and hd["magic"] == 0x3631444D
    assert torch.equal(_values(p, 4096).float(), torch.zeros(4096, device="cuda"))
    spec = SMALL["olmo_s"]
    inp = make_inputs(spec, "cuda")
    inp["W_down"][1, 7, 3] = float("inf")
    layer = run_layer(spec, inp)
    assert _header(layer.down["W_down"])["flags"] == 1
    assert layer.status() == RANGE


@pytest.mark.parametrize("name", BF16_CASES)
@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_kernels_follow_their_rounding(name, fmt):
    """y of each format against Eq. 80 in float64 with h rounded to that format (and, for
    fp16, the expert outputs f and g as well), by the rms of the difference relative to
    rms(y).  The device forms h and f in fp32 (relative error about 2e-6), so about
    2e-6 / ulp of the h elements (and, for fp16, of f and g) round the other way than in the
    emulation, each by one ulp: an rms difference of about 2e-4 for bf16 h, and 1-2e-4
    measured for fp16 h, f and g.  The bars sit well below what rounding h to bf16 would
    give in the fp16 format (1.6e-3)."""
    spec = SMALL[name]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp, h_format=fmt)
    assert layer.status() == 0
    hin = host(inp)
    rt = check_routing_exact(layer, spec)
    tokens = np.arange(spec.T)
    y = layer.out["y"].cpu().double().numpy()
    y_emu = (emulated_y(spec, hin, rt, tokens, torch.float16, torch.float16) if fmt == "f16"
             else emulated_y(spec, hin, rt, tokens, torch.bfloat16))
    err_emu = float(np.sqrt(((y - y_emu) ** 2).mean() / (y_emu ** 2).mean()))
    bar = 4e-4 if fmt == "f16" else 6e-4
    assert err_emu <= bar, f"{name} {fmt}: rms difference from its own rounding {err_emu:.3e}"
    if fmt == "bf16":
        # the optional bf16 intermediate against the oracle, reported beside the bar
        y_ref, _ = oracle_y(spec, hin, rt, tokens)
        record_error(f"{name} (bf16 h, reported only)",
                     layer_error(spec, y, y_ref, rt.route_pos), TOL["bf16"])


def test_h_past_fp16_range_reported_and_scale_restores_it():
    spec = SMALL["olmo_s"]
    inp = make_inputs(spec, "cuda")
    inp["x"] = (inp["x"].float() * 256.0).to(torch.bfloat16)   # exact: a power of two
    layer = run_layer(spec, inp)
    assert layer.status() == RANGE
    assert moe.moe_read_status(layer.ws) == 0                   # read clears it
    layer = run_layer(spec, inp, h_scale_log2=12)
    assert layer.status() == 0
    hin = host(inp)
    rt = check_routing_exact(layer, spec)
    y_ref, _ = oracle_y(spec, hin, rt, np.arange(spec.T))
    err = layer_error(spec, layer.out["y"].cpu().double().numpy(), y_ref, rt.route_pos)
    record_error("olmo_s, x * 256, h_scale_log2 = 12", err, TOL["bf16"])
    assert err <= TOL["bf16"]


def test_bad_pack_reported():
    spec = SMALL["dsv3_s"]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp)
    assert layer.status() == 0
    y0 = layer.out["y"].clone()
    good = dict(layer.down)
    # a buffer of the right size that no pack wrote (zero header)
    layer.down = {"W_down": torch.zeros_like(good["W_down"]), "Ws_down": good["Ws_down"]}
    layer.w = layer._weights(layer.down)
    layer.forward(inp["x"])
    assert layer.status() == BAD_PACK
    # a packed tensor of another size (larger, so every read stays inside it)
    big = torch.cat([inp["W_down"].reshape(-1), inp["W_down"].reshape(-1)[:64]])
    layer.down = {"W_down": moe.pack_weights(big), "Ws_down": good["Ws_down"]}
    layer.w = layer._weights(layer.down)
    layer.forward(inp["x"])
    assert layer.status() == BAD_PACK
    # the right buffers again: the same result as before
    layer.down = good
    layer.w = layer._weights(good)
    y1 = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y1, y0)
