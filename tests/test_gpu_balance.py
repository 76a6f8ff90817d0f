"""Aux-loss-free selection bias (Eq. 35), the bias controller (Eq. 36-37) and the
load-balancing statistics (Eq. 22, 27, 30, 38, 39; entropy deficit), on a GB300,
against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_helpers import (TOL, check_routing_exact, host, layer_error, oracle_y, record_error,
                               run_layer)
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

C = CONFIGS
SHAPES = {
    "tiny": C["tiny"],                                                          # CUDA-core router
    "dsv3_s": C["dsv3"].replace(T=600, d_model=448, d_expert=128, d_shared=128),  # sigmoid, tensor cores
    "olmo_s": C["olmo"].replace(T=1000, d_model=512, d_expert=384, d_shared=256),
    "mixtral_s": C["mixtral"].replace(T=900, d_model=4096, d_expert=1024),     # selected softmax, capacity
}


def _bias(N, scale, seed=3):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(N, generator=g) * scale).to("cuda")


@pytest.mark.parametrize("name", list(SHAPES))
def test_selection_bias_moves_selection_only(name):
    spec = SHAPES[name]
    inp = make_inputs(spec, "cuda")
    b = _bias(spec.N, 0.75)
    inp["selection_bias"] = b
    layer = run_layer(spec, inp)
    assert layer.status() == 0
    rt = check_routing_exact(layer, spec, selection_bias=b)
    # the bias changed some selections, and the weights are those of the unbiased logits
    rt0 = O.route(layer.out["logits"].cpu().numpy(), spec)
    assert (rt.topk_idx != rt0.topk_idx).any()
    hin = host(inp)
    y_ref, _ = oracle_y(spec, hin, rt, np.arange(spec.T))
    err = layer_error(spec, layer.out["y"].cpu().double().numpy(), y_ref, rt.route_pos)
    record_error(f"{name} with selection bias", err, TOL[spec.dtype])
    assert err <= TOL[spec.dtype]


@pytest.mark.parametrize("name", list(SHAPES))
def test_balance_statistics(name):
    import routing_shared_expert_gb300 as moe
    spec = SHAPES[name]
    inp = make_inputs(spec, "cuda")
    layer = run_layer(spec, inp)
    o = layer.out
    P = torch.empty(spec.N, dtype=torch.float32, device="cuda")
    f = torch.empty(spec.N, dtype=torch.float32, device="cuda")
    st = torch.empty(len(moe.STATS), dtype=torch.float32, device="cuda")
    moe.moe_balance_stats(layer.cfg, o["logits"], o["counts_req"], o["counts_keep"], o["R_req"],
                          o["R_keep"], P, f, st, layer.ws)
    torch.cuda.synchronize()
    rt = check_routing_exact(layer, spec)
    p = O.normalized_scores(o["logits"].cpu().numpy(), spec.score)
    f_ref, P_ref, L_ref = O.lbl_statistics(p, rt.topk_idx, spec.N)
    np.testing.assert_allclose(P.cpu().numpy(), P_ref, rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(f.cpu().numpy(), f_ref, rtol=1e-6)
    s = dict(zip(moe.STATS, st.cpu().numpy().tolist()))
    assert abs(s["lbl"] - L_ref) <= 1e-5 * L_ref
    assert abs(s["imax_req"] - O.max_mean_imbalance(rt.counts_req)) < 1e-5
    assert abs(s["imax_keep"] - O.max_mean_imbalance(rt.counts_keep)) < 1e-5
    assert abs(s["imax_rank_req"] - O.max_mean_imbalance(rt.R_req)) < 1e-5
    assert abs(s["imax_rank_keep"] - O.max_mean_imbalance(rt.R_keep)) < 1e-5
    assert abs(s["ih_req"] - O.entropy_deficit(rt.counts_req)) < 1e-5
    assert abs(s["ih_keep"] - O.entropy_deficit(rt.counts_keep)) < 1e-5
    assert abs(s["cv_req"] - O.coefficient_of_variation(rt.counts_req)) < 1e-5
    assert s["never_selected"] == O.never_selected(rt.counts_req)
    assert abs(s["drop_fraction"] - rt.drops["delta_route"]) < 1e-6


def test_bias_update_matches_oracle_bit_for_bit():
    import routing_shared_expert_gb300 as moe
    g = torch.Generator().manual_seed(11)
    for N in (8, 60, 256):
        # counts whose mean is exactly m = 25: n0 experts at m (sign 0 in Eq. 37), the rest in
        # pairs m + delta, m - delta (sign -1 and +1)
        m = 25
        n0 = N // 8 + (N - N // 8) % 2
        delta = torch.randint(1, m + 1, ((N - n0) // 2,), generator=g, dtype=torch.int32)
        counts = torch.cat([torch.full((n0,), m, dtype=torch.int32), m + delta, m - delta])
        counts = counts[torch.randperm(N, generator=g)]
        assert int(counts.sum()) == m * N
        bias = torch.randn(N, generator=g)
        want = O.bias_update(bias.numpy(), counts.numpy(), 0.001)
        b = bias.to("cuda")
        moe.moe_bias_update(N, counts.to("cuda"), 0.001, b)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(b.cpu().numpy(), want)


def test_bias_controller_feedback_loop_balances_requests():
    """Eq. 35-37 closed loop on a skewed router: repeated batches with the post-batch sign update
    reduce the requested max/mean imbalance, and every step matches the oracle exactly."""
    import routing_shared_expert_gb300 as moe
    spec = C["mixtral"].replace(T=1024, d_model=256, d_expert=128, cap_policy="none",
                                capacity_factor=1.0)
    inp = make_inputs(spec, "cuda")
    b = torch.zeros(spec.N, dtype=torch.float32, device="cuda")
    inp["selection_bias"] = b
    layer = moe.MoELayer(moe.config_from_spec(spec), inp, "cuda")
    first = last = None
    for step in range(40):
        layer.forward(inp["x"])
        torch.cuda.synchronize()
        counts = layer.out["counts_req"].cpu().numpy()
        imax = O.max_mean_imbalance(counts)
        first = imax if first is None else first
        last = imax
        before = b.cpu().numpy().copy()
        moe.moe_bias_update(spec.N, layer.out["counts_req"], 0.05, b)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(b.cpu().numpy(), O.bias_update(before, counts, 0.05))
    assert last < 0.6 * first, (first, last)


@pytest.mark.parametrize("N,T,K,M,score", [
    (1, 65, 1, 1, "softmax"), (2, 1, 1, 2, "sigmoid"), (3, 129, 2, 3, "softmax"),
    (5, 700, 2, 2, "sigmoid"), (8, 4100, 2, 8, "softmax"), (12, 63, 3, 4, "sigmoid"),
    (17, 1000, 4, 1, "softmax"), (33, 257, 4, 5, "sigmoid"), (60, 2049, 4, 6, "softmax"),
    (100, 64, 6, 7, "sigmoid"), (200, 3000, 8, 16, "softmax"), (256, 9000, 8, 256, "sigmoid"),
])
def test_balance_statistics_widths(N, T, K, M, score):
    """moe_balance_stats alone on seeded logits and routings of every lane mapping of the score
    pass (1 to 32 lanes per token, 1 to 8 experts per lane), ragged last tiles and T below one
    tile, against the oracle's statistics."""
    import routing_shared_expert_gb300 as moe
    rng = np.random.default_rng(N * 1000 + T)
    z = (rng.standard_normal((T, N)) * 2.0).astype(np.float32)
    # top-K sets drawn with a skew, some experts never chosen when N is large
    w = rng.gamma(0.5, size=N)
    w[rng.random(N) < 0.1] = 0.0
    w = (w + 1e-12) / (w + 1e-12).sum()
    idx = np.stack([rng.choice(N, size=K, replace=False, p=w) for _ in range(T)]).astype(np.int64)
    req = np.bincount(idx.ravel(), minlength=N).astype(np.int32)
    # kept counts: at least one route of every requested expert (the oracle's I_max and I_H
    # are defined for a nonzero load vector)
    keep = np.maximum((req * rng.uniform(0.5, 1.0, N)).astype(np.int32), np.minimum(req, 1))
    rho = np.arange(N) % M
    R_req = np.bincount(rho, weights=req, minlength=M).astype(np.int32)
    R_keep = np.bincount(rho, weights=keep, minlength=M).astype(np.int32)
    cfg = moe.make_config(T=T, d_model=64, N=N, K=K, d_expert=128, d_shared=0, dtype="f32",
                          score=score, shared_mode="none", num_ranks=M, rho=rho.tolist())
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    moe.moe_workspace_init(ws)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    P = torch.empty(N, dtype=torch.float32, device="cuda")
    f = torch.empty(N, dtype=torch.float32, device="cuda")
    st = torch.empty(len(moe.STATS), dtype=torch.float32, device="cuda")
    moe.moe_balance_stats(cfg, dev(z), dev(req), dev(keep), dev(R_req), dev(R_keep), P, f, st, ws)
    torch.cuda.synchronize()
    p = O.normalized_scores(z.astype(np.float64), score)
    f_ref, P_ref, L_ref = O.lbl_statistics(p, idx, N)
    np.testing.assert_allclose(P.cpu().numpy(), P_ref, rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(f.cpu().numpy(), f_ref, rtol=1e-6)
    s = dict(zip(moe.STATS, st.cpu().numpy().tolist()))
    assert abs(s["lbl"] - L_ref) <= 1e-5 * L_ref
    assert abs(s["imax_req"] - O.max_mean_imbalance(req)) < 1e-5
    assert abs(s["imax_keep"] - O.max_mean_imbalance(keep)) < 1e-5
    assert abs(s["imax_rank_req"] - O.max_mean_imbalance(R_req)) < 1e-5
    assert abs(s["imax_rank_keep"] - O.max_mean_imbalance(R_keep)) < 1e-5
    assert abs(s["ih_req"] - O.entropy_deficit(req)) < 1e-5
    assert abs(s["ih_keep"] - O.entropy_deficit(keep)) < 1e-5
    assert abs(s["cv_req"] - O.coefficient_of_variation(req)) < 1e-5
    assert s["never_selected"] == O.never_selected(req)
    assert abs(s["drop_fraction"] - (req.sum() - keep.sum()) / (K * T)) < 1e-6
