"""The seeded synthetic input recipe (no layer arithmetic): determinism, per-tensor seeding,
the init scales of both recipes, and the logit bias profiles.

Recipe: x ~ N(0, 1); weights ~ N(0, 0.02^2) ("0.02" layers) or N(0, 1/fan_in) ("fan_in"
layers: fan_in = d for W_router, W_gate, W_up, w_s; d_r for W_down; the merged width d_s for
the shared W_down); the Qwen2-shaped layer adds an N(0, 1) logit bias per expert and the
Mixtral-shaped layer a Zipf(1.2) profile b_i = -1.2 ln(i + 1); bf16 layers store the fp32
draws rounded to bf16.
"""
import math

import numpy as np
import torch

from workloads import CONFIGS, make_inputs, zipf_logit_bias

SMALL_OLMO = CONFIGS["olmo"].replace(T=512, d_model=256, N=8, d_expert=128, d_shared=64)


def _std(t):
    return float(t.float().std())


def test_same_seed_same_tensors_and_dtype():
    a, b = make_inputs(SMALL_OLMO, "cpu"), make_inputs(SMALL_OLMO, "cpu")
    for k, v in a.items():
        if v is None:
            assert b[k] is None
        else:
            assert v.dtype == (torch.float32 if k == "router_bias" else torch.bfloat16)
            assert torch.equal(v, b[k]), k
    c = make_inputs(SMALL_OLMO, "cpu", seed=1)
    assert not torch.equal(a["x"], c["x"])


def test_each_tensor_seeded_on_its_own():
    """Changing one tensor's shape leaves the others' values unchanged."""
    a = make_inputs(SMALL_OLMO, "cpu")
    b = make_inputs(SMALL_OLMO.replace(d_expert=192, d_shared=128), "cpu")
    assert torch.equal(a["x"], b["x"]) and torch.equal(a["W_router"], b["W_router"])
    assert torch.equal(make_inputs(SMALL_OLMO.replace(T=256), "cpu")["W_up"], a["W_up"])


def test_init_scales_of_both_recipes():
    a = make_inputs(SMALL_OLMO, "cpu")          # "0.02" recipe
    assert abs(_std(a["x"]) - 1.0) < 0.02
    for k in ("W_router", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        assert abs(_std(a[k]) / 0.02 - 1.0) < 0.05, k
    tiny = CONFIGS["tiny"]                      # "fan_in" recipe, fp32, shared split 24+24+16
    t = make_inputs(tiny, "cpu", with_shared_parts=True)
    assert t["x"].dtype == torch.float32
    d, dr, ds = tiny.d_model, tiny.d_expert, tiny.d_shared
    for k, fan in (("W_router", d), ("W_gate", d), ("W_up", d), ("W_down", dr),
                   ("Ws_gate", d), ("Ws_up", d), ("Ws_down", ds)):
        assert abs(_std(t[k]) * math.sqrt(fan) - 1.0) < 0.08, k
    # the merged shared expert is the plain concatenation of its parts
    parts = t["Ws_parts"]
    assert [p[0].shape[0] for p in parts] == list(tiny.shared_split)
    assert torch.equal(t["Ws_gate"], torch.cat([p[0] for p in parts], 0))
    assert torch.equal(t["Ws_down"], torch.cat([p[2] for p in parts], 1))


def test_olmo_router_logit_scale_near_one():
    """Olmo-shaped router: logit std 0.02 * sqrt(2560) ~ 1.0, i.i.d. across experts."""
    cfg = CONFIGS["olmo"].replace(T=256, d_expert=64, d_shared=0, N=32)
    inp = make_inputs(cfg, "cpu")
    z = inp["x"].double() @ inp["W_router"].double().T
    assert abs(float(z.std()) / (0.02 * math.sqrt(2560)) - 1.0) < 0.08
    per_expert_mean = z.mean(0)
    assert float(per_expert_mean.abs().max()) < 0.35   # no per-expert offset


def test_logit_bias_profiles():
    q = make_inputs(CONFIGS["qwen2"].replace(T=64, d_model=128, d_expert=64, d_shared=64), "cpu")
    assert q["router_bias"].dtype == torch.float32 and q["router_bias"].shape == (60,)
    assert abs(_std(q["router_bias"]) - 1.0) < 0.3
    b = zipf_logit_bias(8, 1.2).double().numpy()
    assert np.allclose(b, [-1.2 * math.log(i + 1) for i in range(8)])
    shares = np.exp(b) / np.exp(b).sum()
    assert np.allclose(shares, [0.429, 0.187, 0.115, 0.081, 0.062, 0.050, 0.041, 0.035], atol=1e-3)
    m = make_inputs(CONFIGS["mixtral"].replace(T=64, d_model=128, d_expert=64), "cpu")
    assert torch.equal(m["router_bias"], zipf_logit_bias(8, 1.2))
    assert m["Ws_gate"] is None and m["shared_gate_w"] is None
