"""Pins of the oracle to facts outside itself (CPU only).

Each test checks the oracle against a value the pages print, an identity the
pages state, a closed form worked by hand, or brute force on a tiny input.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.conftest import read_golden
from workloads import CONFIGS, make_inputs


class Cfg:
    """A minimal routing recipe for the oracle's ``route``."""

    def __init__(self, **kw):
        self.__dict__.update(dict(score="softmax", norm="l1", alpha=1.0, cap_policy="none",
                                  capacity_factor=1.0, num_ranks=1, shared_mode="const",
                                  shared_gain=1.0, d_shared=0))
        self.__dict__.update(kw)


# ---------------------------------------------------------------- Figure 69 ---

def test_fig69_olmo_rule_worked_example():
    """Figure 69: p = (.28, .22, .30, .20), K = 4 -> r = K p, sum 4, a_w = 1, sum p^2, R_var."""
    g = read_golden("fig69_merge_example.txt")
    K = int(g["K"][0])
    p = np.array(g["p"])
    # Feed logits ln p for N = K = 4 experts through selection, softmax, L1 and alpha = K.
    z = np.log(p)[None, :]
    cfg = Cfg(N=4, K=K, T=1, alpha=float(K))
    rt = O.route(z, cfg)
    # slot order is by descending logit: (2, 0, 1, 3)
    assert rt.topk_idx[0].tolist() == [2, 0, 1, 3]
    r_by_expert = np.zeros(4)
    r_by_expert[rt.topk_idx[0]] = rt.topk_w[0]
    np.testing.assert_allclose(r_by_expert, g["r"], rtol=0, atol=1e-12)
    assert abs(r_by_expert.sum() - g["sum_r"][0]) < 1e-12
    s = g["s"][0]
    d_r, d_s = int(g["d_r"][0]), int(g["d_s"][0])
    assert round(O.width_weighted_mean(r_by_expert, s, d_r, d_s), 3) == g["a_w"][0]
    assert round(float((p ** 2).sum()), 4) == g["sum_p2"][0]
    assert round(O.variance_ratio(r_by_expert, s, d_r, d_s), 3) == g["R_var"][0]


def test_olmo_invariants_random_tokens():
    """Eq. 83-84: under r = K p the routed coefficients sum to K (mean 1) and a_w = 1 for every token."""
    rng = np.random.default_rng(1)
    for N, K in [(8, 2), (32, 4), (256, 8), (5, 5)]:
        z = rng.normal(size=(64, N))
        rt = O.route(z, Cfg(N=N, K=K, T=64, alpha=float(K)))
        np.testing.assert_allclose(rt.topk_w.sum(1), K, rtol=1e-13)
        for t in range(4):
            assert abs(O.width_weighted_mean(rt.topk_w[t], 1.0, 2560, 1280) - 1.0) < 1e-13


# ------------------------------------------------------------ Eq. 19 / 20 ----

def test_eq19_eq20_count_identities():
    """Eq. 19: sum_i C_i^req = K T.  Eq. 20: destination totals sum to the same routes."""
    rng = np.random.default_rng(2)
    T, N, K, M = 300, 16, 3, 4
    z = rng.normal(size=(T, N))
    rt = O.route(z, Cfg(N=N, K=K, T=T, num_ranks=M))
    assert rt.counts_req.sum() == K * T
    assert rt.R_req.sum() == K * T
    rho = [i % M for i in range(N)]
    for q in range(M):
        assert rt.R_req[q] == sum(rt.counts_req[i] for i in range(N) if rho[i] == q)
    # brute force: count by enumerating (token, expert) pairs
    brute = np.zeros(N, int)
    for t in range(T):
        for e in range(N):
            brute[e] += int(e in set(rt.topk_idx[t].tolist()))
    assert brute.tolist() == rt.counts_req.tolist()


# ---------------------------------------------------------------- Figure 41 ---

def _fig41_idx(requests):
    idx = []
    for e, n in enumerate(requests):
        idx += [e] * n
    return np.array(idx)[:, None]


def test_fig41_capacity_policies():
    """Figure 41 / Eq. 28: per-expert budgets keep 10 and drop 2 (on E0); a shared rank budget keeps all 12."""
    g = read_golden("fig41_capacity_example.txt")
    req = [int(v) for v in g["requests"]]
    rho = [int(v) for v in g["rho"]]
    T, K, N = int(g["T"][0]), int(g["K"][0]), int(g["N"][0])
    c = g["capacity_factor"][0]
    idx = _fig41_idx(req)
    C_req = O.requested_counts(idx, N)
    assert C_req.tolist() == req
    assert O.capacity_limits("per_expert", c, K, T, N) == int(g["b"][0])
    assert O.capacity_limits("rank_wide", c, K, T, N, num_ranks=2) == int(g["B"][0])

    keep_e = O.kept_counts(C_req, "per_expert", c, K, T, rho, 2)
    assert keep_e.tolist() == [int(v) for v in g["per_expert_kept"]]
    assert keep_e.sum() == g["per_expert_kept_total"][0]
    assert (C_req - keep_e).sum() == g["per_expert_dropped_total"][0]

    keep_r = O.kept_counts(C_req, "rank_wide", c, K, T, rho, 2)
    assert keep_r.tolist() == [int(v) for v in g["rank_wide_kept"]]
    assert keep_r.sum() == g["rank_wide_kept_total"][0]
    assert (C_req - keep_r).sum() == g["rank_wide_dropped_total"][0]

    B, b = int(g["B"][0]), int(g["b"][0])
    for q, (d_rank_gold, d_exp_gold) in enumerate(zip(g["rank_wide_D_by_rank"], g["per_expert_D_by_rank"])):
        local = [req[i] for i in range(N) if rho[i] == q]
        d_rank, d_exp = O.drop_totals(local, B, [b] * len(local))
        assert d_rank == d_rank_gold and d_exp == d_exp_gold

    # Eq. 26: rank 0's kept local counts (5, 1) give offsets (5, 6); the oracle's
    # global offsets start each expert's segment at the running sum.
    _, _, offs = O.pack_routes(idx, keep_r, N)
    assert offs[1:3].tolist() == [int(v) for v in g["rank0_rank_wide_offsets"]]


def test_eq29_shared_budget_never_drops_more():
    """Eq. 29: with matched aggregate budgets, D^rank <= D^expert, strict when a neighbour leaves rows unused."""
    rng = np.random.default_rng(3)
    strict = 0
    for _ in range(500):
        n = rng.integers(1, 6)
        b = rng.integers(0, 8, size=n)
        C = rng.integers(0, 12, size=n)
        d_rank, d_exp = O.drop_totals(C, int(b.sum()), b)
        assert d_rank <= d_exp
        strict += d_rank < d_exp
    assert strict > 0


def test_capacity_keeps_token_order_prefix_bruteforce():
    """Per-expert and rank-wide capacity on small random batches, checked against brute force."""
    rng = np.random.default_rng(4)
    for policy in ("per_expert", "rank_wide"):
        for trial in range(20):
            T, N, K, M = int(rng.integers(1, 40)), 6, 2, 3
            z = rng.normal(size=(T, N)) + np.array([2.0, 1.0, 0, 0, 0, -1])  # skewed
            c = float(rng.choice([0.5, 0.75, 1.0, 1.5]))
            rt = O.route(z, Cfg(N=N, K=K, T=T, cap_policy=policy, capacity_factor=c, num_ranks=M))
            rho = [i % M for i in range(N)]
            # budgets by the Eq. 23 / 25 readings
            if policy == "per_expert":
                cap = max(1, math.ceil(c * K * T / N))
                assert (rt.counts_keep == np.minimum(rt.counts_req, cap)).all()
            else:
                B = max(1, math.ceil(c * K * T / M))
                assert (rt.R_keep <= B).all()
                for q in range(M):
                    assert rt.R_keep[q] == min(B, rt.R_req[q])
            # brute force: walk tokens in order, keep while the expert's kept count is below C_keep
            seen = [0] * N
            for t in range(T):
                for k in range(K):
                    e = rt.topk_idx[t, k]
                    assert (rt.route_pos[t, k] >= 0) == (seen[e] < rt.counts_keep[e])
                    seen[e] += 1
            # packed layout: every kept route has a distinct row inside its expert's segment,
            # rows ascend with the token, and perm_src points back at the token.
            pos = rt.route_pos[rt.route_pos >= 0]
            assert sorted(pos.tolist()) == list(range(int(rt.counts_keep.sum())))
            for e in range(N):
                lo, hi = rt.offsets[e], rt.offsets[e + 1]
                toks = rt.perm_src[lo:hi]
                assert (np.diff(toks) > 0).all()
                for t in toks:
                    assert e in rt.topk_idx[t]
            st = rt.drops
            assert abs(st["delta_route"] - (rt.counts_req - rt.counts_keep).sum() / (K * T)) < 1e-15


# ------------------------------------------------------- Eq. 81: dense MLP ---

def test_eq81_dense_reduction():
    """Eq. 81-83: equal logits + the Olmo rule give S = {0..K-1}, r = 1, and the layer is one
    dense SwiGLU over the concatenated blocks of experts 0..K-1 and the shared expert."""
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg, "cpu")
    inp["W_router"] = torch.zeros_like(inp["W_router"])
    y, rt, s = O.moe_forward(cfg, inp)
    K = cfg.K
    assert (rt.topk_idx == np.arange(K)[None, :]).all()
    np.testing.assert_allclose(rt.topk_w, 1.0, rtol=1e-15)
    # one dense SwiGLU with d_act = K d_r + d_s columns (Eq. 81), built by concatenation
    Wg = np.concatenate([O.f64(inp["W_gate"][e]) for e in range(K)] + [O.f64(inp["Ws_gate"])], 0)
    Wu = np.concatenate([O.f64(inp["W_up"][e]) for e in range(K)] + [O.f64(inp["Ws_up"])], 0)
    Wd = np.concatenate([O.f64(inp["W_down"][e]) for e in range(K)] + [O.f64(inp["Ws_down"])], 1)
    assert Wg.shape[0] == K * cfg.d_expert + cfg.d_shared       # Eq. 82 analogue
    x = O.f64(inp["x"])
    a = x @ Wg.T
    dense = ((a / (1 + np.exp(-a))) * (x @ Wu.T)) @ Wd.T
    err = np.abs(y - dense).max() / np.sqrt((dense ** 2).mean())
    assert err < 1e-12


# ---------------------------------------------------- Eq. 75-76: shared merge --

def test_eq76_ungated_shared_experts_merge():
    """Eq. 75-76: three ungated shared experts (24 + 24 + 16) sum to the merged width-64 expert."""
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg, "cpu", with_shared_parts=True)
    parts = inp["Ws_parts"]
    assert [p[0].shape[0] for p in parts] == list(cfg.shared_split)
    x = inp["x"]
    summed = sum(O.swiglu(x, *p) for p in parts)
    Wg, Wu, Wd = O.merge_shared(parts)
    assert Wg.shape == (cfg.d_shared, cfg.d_model) and Wd.shape == (cfg.d_model, cfg.d_shared)
    np.testing.assert_array_equal(Wg, O.f64(inp["Ws_gate"]))
    np.testing.assert_array_equal(Wd, O.f64(inp["Ws_down"]))
    merged = O.swiglu(x, Wg, Wu, Wd)
    rel = np.abs(summed - merged).max() / np.sqrt((merged ** 2).mean())
    assert rel < 1e-12
    # Eq. 77: one common gate a(x) on the sum equals the gate on the merged expert
    a = np.linspace(0.1, 0.9, x.shape[0])[:, None]
    assert np.abs(a * summed - a * merged).max() < 1e-12


# ------------------------------------------------- Table 52 routed mass etc. --

def test_routed_mass_below_one_without_renormalisation():
    """Table 52: top-K of a full softmax without renormalisation keeps m_K < 1 (K < N); = 1 when K = N."""
    rng = np.random.default_rng(5)
    z = rng.normal(size=(200, 60)) * 3
    rt = O.route(z, Cfg(N=60, K=4, T=200, norm="none"))
    m = rt.topk_w.sum(1)
    assert (m > 0).all() and (m < 1).all()
    rt = O.route(z[:, :4], Cfg(N=4, K=4, T=200, norm="none"))
    np.testing.assert_allclose(rt.topk_w.sum(1), 1.0, rtol=1e-14)


def test_softmax_selected_equals_l1_on_full_softmax_and_sigmoid_sums():
    """Table 52: softmax over the selected logits equals L1-renormalised full-softmax probabilities;
    L1-renormalised sigmoid affinities sum to one, so r sums to alpha (2.5 for the DeepSeek-V3 rule)."""
    rng = np.random.default_rng(6)
    z = rng.normal(size=(100, 8)) * 2
    idx = O.select_topk(z, 2)
    a = O.selected_weights(z, idx, "softmax", "softmax_selected")
    b = O.selected_weights(z, idx, "softmax", "l1")
    np.testing.assert_allclose(a, b, rtol=1e-13)
    z = rng.normal(size=(100, 256))
    rt = O.route(z, Cfg(N=256, K=8, T=100, score="sigmoid", norm="l1", alpha=2.5))
    np.testing.assert_allclose(rt.topk_w.sum(1), 2.5, rtol=1e-14)
    # the selected sigmoid affinities are the 8 largest sigma(z)
    q = 1 / (1 + np.exp(-z))
    for t in range(5):
        assert set(rt.topk_idx[t].tolist()) == set(np.argsort(-q[t])[:8].tolist())


def test_lp_normalisation_pins():
    """Table 52, MegaBlocks row: the selected weights may receive an L_p normalisation.
    A 3-4-5 triangle by hand: softmax over logits (ln 3, ln 4, ln 1) gives q = (3, 4, 1) / 8;
    the top 2 in slot order are experts 1, 0 and their L2-normalised weights are 4/5, 3/5."""
    z = np.log(np.array([[3.0, 4.0, 1.0]]))
    idx = O.select_topk(z, 2)
    assert idx.tolist() == [[1, 0]]
    w = O.selected_weights(z, idx, "softmax", "lp", p=2.0)
    np.testing.assert_allclose(w[0], [0.8, 0.6], rtol=1e-14)
    # p = 3 on selected sigmoid scores sigma(ln 3) = 3/4 and sigma(ln 1) = 1/2, by hand:
    # ||(3/4, 1/2)||_3 = (27/64 + 8/64)^(1/3) = (35/64)^(1/3)
    z = np.log(np.array([[3.0, 1.0]]))
    w = O.selected_weights(z, np.array([[0, 1]]), "sigmoid", "lp", p=3.0)
    n = (35.0 / 64.0) ** (1.0 / 3.0)
    np.testing.assert_allclose(w[0], [0.75 / n, 0.5 / n], rtol=1e-14)
    rng = np.random.default_rng(11)
    z = rng.normal(size=(200, 32))
    idx = O.select_topk(z, 4)
    q = np.take_along_axis(O.softmax_all(z), idx, axis=1)
    # p = 1 is the L1 rule
    np.testing.assert_allclose(O.selected_weights(z, idx, "softmax", "lp", p=1.0),
                               O.selected_weights(z, idx, "softmax", "l1"), rtol=1e-14)
    for pp in (1.5, 2.0, 3.0, 8.0):
        w = O.selected_weights(z, idx, "softmax", "lp", p=pp)
        # unit L_p norm, and a per-token rescaling of the scores (ratios kept)
        np.testing.assert_allclose((w ** pp).sum(1), 1.0, rtol=1e-13)
        np.testing.assert_allclose(w / w[:, :1], q / q[:, :1], rtol=1e-13)
    # towards L_inf: K^(-1/p) <= max_k w_k <= 1
    w = O.selected_weights(z, idx, "softmax", "lp", p=200.0)
    assert np.all(w.max(1) <= 1 + 1e-15) and np.all(w.max(1) >= 4 ** (-1 / 200) - 1e-15)
    # through route(): r = alpha w with the config's p
    rt = O.route(z, Cfg(N=32, K=4, T=200, norm="lp", norm_p=2.0, alpha=4.0))
    np.testing.assert_allclose((rt.topk_w ** 2).sum(1), 16.0, rtol=1e-13)


def test_sigmoid_and_softmax_closed_forms():
    assert O.sigmoid(np.array([[0.0]]))[0, 0] == 0.5
    assert abs(O.sigmoid(np.array([[math.log(3.0)]]))[0, 0] - 0.75) < 1e-15
    q = O.softmax_all(np.log(np.array([[1.0, 2.0, 5.0]])))
    np.testing.assert_allclose(q[0], [0.125, 0.25, 0.625], rtol=1e-15)


# ------------------------------------------------------------ brute-force top-K

def test_topk_bruteforce_with_ties():
    """Exactly one K-subset dominates the rest (a_i > a_j, or equal with lower index); it is select_topk's."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        N = int(rng.integers(1, 9))
        K = int(rng.integers(1, N + 1))
        a = rng.integers(-2, 3, size=N).astype(float)      # small integers force ties
        winners = []
        for S in itertools.combinations(range(N), K):
            Sset = set(S)
            if all((a[i] > a[j]) or (a[i] == a[j] and i < j)
                   for i in Sset for j in range(N) if j not in Sset):
                winners.append(S)
        assert len(winners) == 1
        got = O.select_topk(a[None, :], K)[0]
        assert set(got.tolist()) == set(winners[0])
        # slot order: descending key, ascending index among equals
        keys = [(-a[i], i) for i in got]
        assert keys == sorted(keys)


def test_all_equal_logits_select_lowest_indices():
    z = np.zeros((3, 10))
    assert O.select_topk(z, 4).tolist() == [[0, 1, 2, 3]] * 3


# --------------------------------------------------------- six-token example --

def test_eq43_six_token_requested_counts():
    """Eq. 43-44: top-1 over the six-token score table gives C^req = (2, 4) and I_max = 4/3 (Eq. 39)."""
    g = read_golden("eq43_six_token_example.txt")
    scores = np.array(g["scores"])
    idx = O.select_topk(scores, 1)
    C = O.requested_counts(idx, 2)
    assert C.tolist() == [int(v) for v in g["C_req"]]
    f = C / C.sum()
    np.testing.assert_allclose(f, g["f"], rtol=1e-15)
    assert abs(2 * f.max() - g["I_max"][0]) < 1e-15


# ------------------------------------------------- SwiGLU and Eq. 80 by hand --

def _silu(v):
    return v / (1.0 + math.exp(-v))


def test_swiglu_scalar_closed_form():
    """Eq. 74 with d = m = 1: E(x) = SiLU(x w_g) (x w_u) w_d; swapping gate and up changes the value."""
    x, wg, wu, wd = 1.0, 2.0, 3.0, 0.5
    want = _silu(2.0) * 3.0 * 0.5
    got = O.swiglu(np.array([[x]]), np.array([[wg]]), np.array([[wu]]), np.array([[wd]]))[0, 0]
    assert abs(got - want) < 1e-15
    assert abs(want - _silu(3.0) * 2.0 * 0.5) > 0.1
    # non-square shapes: d = 2, m = 3, hand-evaluated
    x = np.array([[1.0, -2.0]])
    Wg = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])       # gate pre-activations (1, -2, -1)
    Wu = np.array([[2.0, 0.0], [0.0, 0.5], [1.0, 0.0]])       # up (2, -1, 1)
    Wd = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, -1.0]])        # [d=2, m=3]
    h = [_silu(1.0) * 2.0, _silu(-2.0) * -1.0, _silu(-1.0) * 1.0]
    want = [h[0] + 2.0 * h[2], h[1] - h[2]]
    np.testing.assert_allclose(O.swiglu(x, Wg, Wu, Wd)[0], want, rtol=1e-15)


def test_eq80_merge_scalar_closed_form():
    """Eq. 80 on a hand-worked token: two scalar experts, softmax router, L1 + alpha = 2, unit shared gain."""
    x = np.array([[1.0]])
    Wg = np.array([[[2.0]], [[-1.0]]])
    Wu = np.array([[[3.0]], [[1.0]]])
    Wd = np.array([[[0.5]], [[1.0]]])
    inputs = dict(x=x, W_router=None, W_gate=Wg, W_up=Wu, W_down=Wd,
                  Ws_gate=np.array([[1.0]]), Ws_up=np.array([[1.0]]), Ws_down=np.array([[1.0]]))
    cfg = Cfg(N=2, K=2, T=1, alpha=2.0, d_shared=1, shared_mode="const", shared_gain=1.0)
    z = np.log(np.array([[3.0, 1.0]]))          # softmax (3/4, 1/4)
    y, rt, s = O.moe_forward(cfg, inputs, logits=z)
    f0 = _silu(2.0) * 3.0 * 0.5
    f1 = _silu(-1.0) * 1.0 * 1.0
    g = _silu(1.0)
    want = 2.0 * 0.75 * f0 + 2.0 * 0.25 * f1 + 1.0 * g
    assert abs(y[0, 0] - want) < 1e-14
    # a dropped route contributes nothing and the survivor is not renormalised
    cfg_cap = Cfg(N=2, K=2, T=1, alpha=2.0, d_shared=1, cap_policy="rank_wide",
                  capacity_factor=0.5, num_ranks=1)
    y2, rt2, _ = O.moe_forward(cfg_cap, inputs, logits=z)
    assert rt2.route_pos[0].tolist() == [0, -1]
    assert abs(y2[0, 0] - (2.0 * 0.75 * f0 + g)) < 1e-14
    assert abs(rt2.drops["removed_weight"] - 0.5) < 1e-15
    assert rt2.drops["tokens_lost_any"] == 1 and rt2.drops["tokens_lost_all"] == 0


def test_shared_gate_closed_form():
    """Eq. 77 / Table 52 (Qwen): s(x) = sigma(w_s . x)."""
    x = np.array([[1.0, 2.0], [0.0, 0.0]])
    w = np.array([0.5, -0.25])      # w.x = 0 and 0
    s = O.shared_coefficient(x, "gate", 1.0, w)
    np.testing.assert_allclose(s, [0.5, 0.5], rtol=0)
    x = np.array([[math.log(3.0), 0.0]])
    s = O.shared_coefficient(x, "gate", 1.0, np.array([1.0, 7.0]))
    assert abs(s[0] - 0.75) < 1e-15


# ----------------------------------------------- Section 10.5-10.7: balancing --

def test_eq45_six_token_lbl(golden):
    """Eq. 43-45: f = (1/3, 2/3), P = (3/5, 2/5), L = 14/15, and the centered form (Eq. 41)."""
    g = read_golden("eq43_six_token_example.txt")
    p = np.array(g["scores"])
    idx = O.select_topk(p, 1)
    f, P, L = O.lbl_statistics(p, idx, 2)
    np.testing.assert_allclose(f, g["f"], rtol=1e-15)
    np.testing.assert_allclose(P, g["P"], rtol=1e-15)
    assert abs(L - g["L_LBL"][0]) < 1e-15
    u = np.full(2, 0.5)
    assert abs(L - (1 + 2 * (f - u) @ (P - u))) < 1e-15
    assert abs(O.max_mean_imbalance(O.requested_counts(idx, 2)) - g["I_max"][0]) < 1e-15


def test_eq40_eq42_lbl_identities():
    """Eq. 42: P = u gives L = 1 for any f; Eq. 40: P = f gives L = 1 + N ||f - u||^2; Eq. 41 in general."""
    rng = np.random.default_rng(8)
    for N, K, T in [(4, 1, 50), (16, 2, 200), (64, 4, 300)]:
        idx = np.stack([rng.choice(N, size=K, replace=False) for _ in range(T)])
        f, _, _ = O.lbl_statistics(np.full((T, N), 1.0 / N), idx, N)
        assert abs(O.lbl_statistics(np.full((T, N), 1.0 / N), idx, N)[2] - 1.0) < 1e-12
        # a score table whose column means equal f
        p = np.tile(f, (T, 1))
        L = O.lbl_statistics(p, idx, N)[2]
        u = np.full(N, 1.0 / N)
        assert abs(L - (1 + N * ((f - u) ** 2).sum())) < 1e-12
        z = rng.normal(size=(T, N))
        p = O.softmax_all(z)
        f, P, L = O.lbl_statistics(p, idx, N)
        assert abs(L - (1 + N * (f - u) @ (P - u))) < 1e-12


def test_eq48_two_expert_infimum(golden):
    """Eq. 47-49: with expert-1 routes scoring (1, 0) and expert-2 routes (1/2 - e, 1/2 + e),
    L approaches 1 - x + 2 x^2 as e -> 0: 7/8 at x = 1/4, 8/9 for the 2:4 split."""
    g = read_golden("eq48_52_lbl_limits.txt")
    for xk, lk in (("two_expert_x", "two_expert_inf"), ("two_expert_x_split", "two_expert_inf_split")):
        x = g[xk][0]
        T = 12
        n1 = int(round(x * T))
        eps = 1e-9
        p = np.array([[1.0, 0.0]] * n1 + [[0.5 - eps, 0.5 + eps]] * (T - n1))
        idx = O.select_topk(p, 1)
        assert (idx[:n1, 0] == 0).all() and (idx[n1:, 0] == 1).all()
        L = O.lbl_statistics(p, idx, 2)[2]
        assert abs(L - g[lk][0]) < 1e-8
        assert abs(g[lk][0] - (1 - x + 2 * x * x)) < 1e-15


def test_eq52_many_expert_limit(golden):
    """Eq. 50-52: A active experts win uniformly; winners score (1 + D e)/(D + K), dead experts
    (1 - K e)/(D + K), other active experts ~0; L -> N K / (A (N - A + K))."""
    g = read_golden("eq48_52_lbl_limits.txt")
    N, A, K = int(g["many_N"][0]), int(g["many_A"][0]), int(g["many_K"][0])
    for (N, A, K, want) in [(N, A, K, g["many_limit"][0]), (64, 16, 4, None), (32, 8, 2, None)]:
        D = N - A
        eps = 1e-10
        T = A * 10
        p = np.zeros((T, N))
        for t in range(T):
            win = [(t * K + j) % A for j in range(K)]
            p[t, A:] = (1 - K * eps) / (D + K)
            p[t, win] = (1 + D * eps) / (D + K)
        idx = O.select_topk(p, K)
        L = O.lbl_statistics(p, idx, N)[2]
        limit = N * K / (A * (N - A + K))
        if want is not None:
            assert abs(limit - want) < 1e-15
        assert abs(L - limit) < 1e-8
        assert abs(O.max_mean_imbalance(O.requested_counts(idx, N)) - N / A) < 1e-12
        assert O.never_selected(O.requested_counts(idx, N)) == D


def test_entropy_deficit_and_cv_closed_forms():
    assert O.entropy_deficit(np.full(8, 5)) == 0.0
    assert O.entropy_deficit(np.array([7])) == 0.0                # one expert: no deficit
    assert abs(O.entropy_deficit(np.eye(8)[3]) - 1.0) < 1e-15
    x = np.array([1, 1, 0, 0])
    assert abs(O.entropy_deficit(x) - 0.5) < 1e-15            # log 2 / log 4
    assert O.coefficient_of_variation(np.full(5, 3)) == 0.0
    assert abs(O.coefficient_of_variation(np.array([0, 2])) - 1.0) < 1e-15
    assert O.max_mean_imbalance(np.full(6, 7)) == 1.0


def test_eq37_bias_update_by_hand():
    """Eq. 36-37: b_i <- b_i + gamma sign(mean C - C_i)."""
    b = O.bias_update(np.array([0.0, 0.5, -0.25, 1.0]), np.array([5, 1, 3, 3]), 0.125)
    np.testing.assert_array_equal(b, np.array([-0.125, 0.625, -0.25, 1.0], np.float32))


def test_eq35_selection_bias_moves_selection_not_weights():
    """Eq. 35: the bias enters the selection key only; weights come from the unbiased logits."""
    z = np.array([[1.0, 0.9, -1.0, 0.0]])
    cfg = Cfg(N=4, K=2, T=1, alpha=1.0)
    plain = O.route(z, cfg)
    assert sorted(plain.topk_idx[0].tolist()) == [0, 1]
    biased = O.route(z, cfg, selection_bias=[0.0, 0.0, 0.0, 1.5])
    assert biased.topk_idx[0].tolist() == [3, 0]           # keys (1.0, 0.9, -1.0, 1.5)
    e = np.exp(np.array([0.0, 1.0]))
    np.testing.assert_allclose(biased.topk_w[0], e / e.sum(), rtol=1e-15)


# ------------------------------- Section 10.7.1: sigmoid scores in the LBL term --

def _sigmoid_lbl_case():
    """Six tokens, two experts, top-1, sigmoid routing.  Two tokens have logits (ln 3, 0),
    so sigma = (3/4, 1/2) and the scores normalised across the experts are (3/5, 2/5); four
    tokens have logits (0, ln 3) and normalised scores (2/5, 3/5).  Expert 0 wins the first
    two tokens, expert 1 the other four: C = (2, 4), f = (1/3, 2/3),
    P = ((2 * 3/5 + 4 * 2/5) / 6, (2 * 2/5 + 4 * 3/5) / 6) = (7/15, 8/15) and
    L = 2 (1/3 * 7/15 + 2/3 * 8/15) = 46/45 (Eq. 30, Eq. 38)."""
    l3 = math.log(3.0)
    z = np.array([[l3, 0.0]] * 2 + [[0.0, l3]] * 4)
    return z, (2, 4), (1 / 3, 2 / 3), (7 / 15, 8 / 15), 46 / 45


def _check_sigmoid_lbl(normalized_scores):
    z, C, f_want, P_want, L_want = _sigmoid_lbl_case()
    p = normalized_scores(z, "sigmoid")
    np.testing.assert_allclose(p[0], [3 / 5, 2 / 5], rtol=1e-14)
    np.testing.assert_allclose(p[2], [2 / 5, 3 / 5], rtol=1e-14)
    # three experts by hand: sigma(ln 3, 0, -ln 3) = (3/4, 1/2, 1/4), sum 3/2
    l3 = math.log(3.0)
    np.testing.assert_allclose(normalized_scores(np.array([[l3, 0.0, -l3]]), "sigmoid")[0],
                               [1 / 2, 1 / 3, 1 / 6], rtol=1e-14)
    idx = O.select_topk(z, 1)
    assert O.requested_counts(idx, 2).tolist() == list(C)
    f, P, L = O.lbl_statistics(p, idx, 2)
    np.testing.assert_allclose(f, f_want, rtol=1e-14)
    np.testing.assert_allclose(P, P_want, rtol=1e-14)
    assert abs(L - L_want) < 1e-14
    # Eq. 38: P is a probability vector for sigmoid routing too
    rng = np.random.default_rng(11)
    zr = rng.normal(size=(40, 7))
    assert abs(O.lbl_statistics(normalized_scores(zr, "sigmoid"), O.select_topk(zr, 2), 7)[1]
               .sum() - 1.0) < 1e-13


def test_section10_7_1_sigmoid_scores_normalised_across_experts():
    """Section 10.7.1: for sigmoid routing the LBL's soft term uses the sigmoid scores divided
    by their sum over the experts of the token; worked by hand on a six-token example."""
    _check_sigmoid_lbl(O.normalized_scores)
    # softmax scores are used as they are (already normalised)
    z = np.array([[0.0, math.log(3.0)]])
    np.testing.assert_allclose(O.normalized_scores(z, "softmax")[0], [1 / 4, 3 / 4], rtol=1e-15)


@pytest.mark.parametrize("mistake", ["unnormalised", "divided_by_N", "softmax_of_sigmoid"])
def test_sigmoid_lbl_pin_catches_plausible_mistakes(mistake):
    """The pin above fails for each plausible misreading of the normalisation (mistakes planted
    in a copy of the oracle function, on the CPU): sigmoid scores left unnormalised
    (L = 23/18), divided by N instead of their sum (L = 23/36), or a softmax over them."""
    def wrong(z, score):
        if score == "softmax":
            return O.softmax_all(z)
        q = O.sigmoid(z)
        if mistake == "unnormalised":
            return q
        if mistake == "divided_by_N":
            return q / q.shape[1]
        return O.softmax_all(q)
    with pytest.raises(AssertionError):
        _check_sigmoid_lbl(wrong)


# ------------------------------------------- the additive per-expert logit bias --

def _bias_layer():
    """One token, d = 1, three experts, K = 2, softmax scores kept without renormalisation
    (the Qwen row of Table 52).  Projection logits x W_r^T = (ln 4, ln 2, 0); the logit bias
    (0, ln 4, 0) makes z = (ln 4, ln 8, 0), whose softmax is (4, 8, 1) / 13."""
    inputs = {
        "x": np.array([[1.0]]),
        "W_router": np.array([[math.log(4.0)], [math.log(2.0)], [0.0]]),
        "router_bias": np.array([0.0, math.log(4.0), 0.0]),
        "W_gate": np.ones((3, 1, 1)), "W_up": np.ones((3, 1, 1)), "W_down": np.ones((3, 1, 1)),
    }
    cfg = Cfg(N=3, K=2, T=1, score="softmax", norm="none", alpha=1.0, shared_mode="none")
    return cfg, inputs


# expected by hand, and what each misreading of the bias would give instead
BIAS_EXPECTED = ([1, 0], [8 / 13, 4 / 13])
BIAS_MISREADINGS = {
    "bias ignored": ([0, 1], [4 / 7, 2 / 7]),
    "bias in the selection only": ([1, 0], [2 / 7, 4 / 7]),
    "bias in the scores only": ([0, 1], [4 / 13, 8 / 13]),
}


def _check_bias(oracle_module, check_logits=True):
    cfg, inputs = _bias_layer()
    if check_logits:
        z = oracle_module.router_logits(inputs["x"], inputs["W_router"], inputs["router_bias"])
        np.testing.assert_allclose(z[0], np.log([4.0, 8.0, 1.0]), rtol=1e-15)
    y, rt, _ = oracle_module.moe_forward(cfg, inputs)
    assert rt.topk_idx[0].tolist() == BIAS_EXPECTED[0]
    np.testing.assert_allclose(rt.topk_w[0], BIAS_EXPECTED[1], rtol=1e-14)
    # routed mass 12/13 < 1 (Table 52, no renormalisation)
    assert abs(rt.topk_w[0].sum() - 12 / 13) < 1e-15
    # experts are identity-like: f_i(1) = SiLU(1) * 1 * 1, so y = (12/13) SiLU(1)
    assert abs(y[0, 0] - 12 / 13 / (1 + math.exp(-1.0))) < 1e-14


def test_logit_bias_enters_selection_and_scores():
    """An additive per-expert logit bias (the Qwen2- and Mixtral-shaped layers' recipe) is part
    of the logit: it moves both the selected set and the softmax weights.  Worked by hand: the
    bias turns the selection from (0, 1) into (1, 0) and the weights into (8/13, 4/13)."""
    _check_bias(O)
    # the hand values of every misreading differ from the expected ones in the selection,
    # the weights, or both, so the pin above rejects each of them
    for idx, w in BIAS_MISREADINGS.values():
        assert idx != BIAS_EXPECTED[0] or not np.allclose(w, BIAS_EXPECTED[1])


def test_logit_bias_pin_catches_a_dropped_bias(monkeypatch):
    """A mistake planted in the oracle on the CPU: a router projection that drops the bias
    fails the pin, both on the logits and through the whole forward."""
    real = O.moe_oracle.router_logits
    monkeypatch.setattr(O.moe_oracle, "router_logits", lambda x, W, b=None: real(x, W, None))
    with pytest.raises(AssertionError):
        _check_bias(O.moe_oracle)
    with pytest.raises(AssertionError):
        _check_bias(O.moe_oracle, check_logits=False)
