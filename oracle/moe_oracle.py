"""Oracle for the forward pass of a routed + shared-expert MoE layer.

TEST INFRASTRUCTURE.  This module is the plain, slow, obviously correct CPU
statement of what the layer computes.  Only the test suite, the smoke check and
the benchmark's CPU-baseline / reference arm may import or run it; the library
(``routing_shared_expert_gb300``) never does, and the two share no code.

Everything is numpy in float64.  bf16 / fp32 inputs are up-converted exactly.
Where a floating-point comparison decides an integer result (the top-K
selection), the comparison is made on the keys exactly as given: callers that
check the device path hand in the device's fp32 router logits, so both sides
decide on the same fp32 values.

Sources (page title, then section / equation / table):

* "Section 21: Merging Routed and Shared Expert Activations" - Eq. 80 (merge
  rule), Eq. 81-82 (dense decomposition), Eq. 83 (Olmo rule r = K p, s = 1),
  Eq. 84 (width-weighted mean), Eq. 85-86 (variance ratio), Fig. 69, Table 37.
* "Appendix E: Expert-Merge Normalization in Public MoE Models" - Table 52
  (selected renormalisation, routed scale alpha, routed mass m_K < 1 without
  renormalisation, softmax over the selected logits, learned sigmoid shared gate,
  sigmoid affinities).
* "Shared and Fine-Grained Experts" - softmax router, top-k, renormalise the k.
* "Section 20: One Shared Expert Is All You Need" - Eq. 74 (SwiGLU expert),
  Eq. 75-76 (merging ungated shared experts), Eq. 77 (one common gate).
* "Section 10: Routing, Capacity, and Load Balancing" - Eq. 19-21 (requested /
  kept counts, destination totals), Eq. 22 (max/mean), Eq. 23 and 25
  (rank-wide and per-expert capacity), Eq. 26 (packed offsets), the admission
  order of Section 10.3, Eq. 27 (route-drop fraction), Eq. 28-29 (drop totals),
  Eq. 35 (selection on logits for softmax routing, selection-only bias),
  Eq. 36-37 (bias controller), Eq. 30 / 38 (load-balancing loss statistics),
  Eq. 39 (requested max/mean), the entropy deficit of Section 10.2.

Readings where the pages are silent or ambiguous are stated beside the code
that takes them.  Every function is pinned by tests/test_oracle_pins.py to values
the pages print, closed forms, brute force or identities; the expert and shared
outputs f_i, g and the merged y by hand-evaluated SwiGLU and Eq. 80 tokens and by
the Eq. 81 dense reduction, written out independently with numpy at a random
layer.  The full layer shapes run the same shape-generic code.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64

SCORES = ("softmax", "sigmoid")
NORMS = ("none", "l1", "softmax_selected", "lp")
SHARED_MODES = ("none", "const", "gate")
CAP_POLICIES = ("none", "per_expert", "rank_wide")


def f64(a) -> np.ndarray:
    """Exact up-conversion of a numpy array or torch tensor (fp32 / bf16) to float64."""
    if hasattr(a, "detach"):          # torch tensor; bf16 has no numpy dtype
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------- #
# Router: logits, selection, scores, coefficients                              #
# --------------------------------------------------------------------------- #

def router_logits(x, W_router, router_bias=None) -> np.ndarray:
    """z_t = x_t W_r (+ b): the router projection ("Section 10", Table 16, first row).

    ``W_router`` is stored one row per expert ([N, d]), so z = x W_router^T.
    Reading: a per-expert logit bias, where a layer has one, is part of the
    logit; it enters both the selection and the scores.
    """
    z = f64(x) @ f64(W_router).T
    if router_bias is not None:
        z = z + f64(router_bias)[None, :]
    return z


def select_topk(keys, K: int) -> np.ndarray:
    """S_t = TopK_i(a_t,i, K) ("Section 10.6", Eq. 35 without bias; "Shared and Fine-Grained Experts").

    Reading (the pages are silent on ties): expert i is selected before j when
    a_i > a_j, or a_i == a_j and i < j.  Slot k of the result holds the k-th
    expert in that order.  For softmax routing the key is the logit z (Eq. 35:
    a = z); for sigmoid affinities the key is also z, since sigma is monotone
    and selects the same set.
    """
    keys = np.asarray(keys)
    if not 1 <= K <= keys.shape[1]:
        raise ValueError("need 1 <= K <= N")
    # A stable sort of -a keeps equal keys in ascending index order.
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :K].astype(np.int64)


def softmax_all(z) -> np.ndarray:
    """q_t = softmax(z_t) over all N experts ("Shared and Fine-Grained Experts": gate(x).softmax)."""
    z = f64(z)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=1, keepdims=True)


def sigmoid(z) -> np.ndarray:
    """sigma(z) = 1 / (1 + exp(-z)), elementwise (sigmoid affinities, "Appendix E", Table 52)."""
    z = f64(z)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def selected_weights(z, idx, score: str, norm: str, p: float = 2.0) -> np.ndarray:
    """Per-slot mixture weights w_t,k before the routed scale ("Appendix E", Table 52).

    * ``none``: w = q_S, the selected scores as they are (routed mass m_K < 1
      for a softmax over N > K experts).
    * ``l1``: w = q_S / sum_{j in S} q_j ("Section 21.1": selected probabilities
      after L1 normalisation; "Shared and Fine-Grained Experts": renormalise the k).
    * ``softmax_selected``: w = softmax(z_S), the softmax over the selected
      logits only (Mixtral row of Table 52).  It does not look at ``score``.
    * ``lp``: w = q_S / ||q_S||_p = q_S / (sum_{j in S} q_j^p)^(1/p), the L_p
      normalisation of the selected weights the MegaBlocks row of Table 52 offers
      (the row names no p; it is a parameter, and p = 1 is ``l1``).
    """
    z = f64(z)
    idx = np.asarray(idx)
    zS = np.take_along_axis(z, idx, axis=1)
    if norm == "softmax_selected":
        m = zS.max(axis=1, keepdims=True)
        e = np.exp(zS - m)
        return e / e.sum(axis=1, keepdims=True)
    q = softmax_all(z) if score == "softmax" else sigmoid(z)
    qS = np.take_along_axis(q, idx, axis=1)
    if norm == "none":
        return qS
    if norm == "l1":
        return qS / qS.sum(axis=1, keepdims=True)
    if norm == "lp":
        return qS / np.power(np.power(qS, p).sum(axis=1, keepdims=True), 1.0 / p)
    raise ValueError(norm)


def shared_coefficient(x, shared_mode: str, shared_gain: float, shared_gate_w=None) -> np.ndarray:
    """s(x) of Eq. 80: 0 without a shared expert, a constant gain, or sigma(w_s . x).

    The learned gate is one scalar per token applied to the whole shared branch
    ("Section 20.1", Eq. 77 a(x) E*(x); "Appendix E", Table 52, Qwen rows).
    """
    T = int(x.shape[0])
    if shared_mode == "none":
        return np.zeros(T, F64)
    if shared_mode == "const":
        return np.full(T, float(shared_gain), F64)
    if shared_mode == "gate":
        u = f64(x) @ f64(shared_gate_w)
        return sigmoid(u[:, None])[:, 0]
    raise ValueError(shared_mode)


# --------------------------------------------------------------------------- #
# Counts, capacity, packing                                                    #
# --------------------------------------------------------------------------- #

def requested_counts(idx, N: int) -> np.ndarray:
    """C_i^req = sum_t 1{i in S_t} ("Section 10.1", Eq. 19)."""
    return np.bincount(np.asarray(idx).ravel(), minlength=N).astype(np.int64)


def destination_totals(C, rho, num_ranks: int) -> np.ndarray:
    """R_q = sum_{i: rho(i) = q} C_i ("Section 10.1", Eq. 20 and Eq. 21)."""
    R = np.zeros(num_ranks, np.int64)
    for i, c in enumerate(np.asarray(C)):
        R[int(rho[i])] += int(c)
    return R


def capacity_limits(policy: str, capacity_factor: float, K: int, T: int, N: int,
                    num_ranks: int = 1):
    """Budgets of the capacity policies ("Section 10.3", Eq. 23 and Eq. 25).

    Reading for one device that holds the whole batch: T_route = K T routes
    come from one source.  Per expert: b = max(1, ceil(c K T / N)) (Eq. 25 with
    N_local = N, with the max(1, .) of Eq. 23).  Rank-wide: the batch is read as
    spread evenly over the M_E ranks of the map rho, so each destination's
    budget is B = max(1, ceil(c K T / M_E)), c times its balanced load (Eq. 23).
    Both reproduce Figure 41 (T = 12, K = 1, N = 4, M_E = 2, c = 1: b = 3, B = 6).
    Returns None without a capacity limit, else the per-expert budget or the
    per-rank budget.
    """
    if policy == "none":
        return None
    if policy == "per_expert":
        return max(1, int(math.ceil(capacity_factor * K * T / N)))
    if policy == "rank_wide":
        return max(1, int(math.ceil(capacity_factor * K * T / num_ranks)))
    raise ValueError(policy)


def kept_counts(C_req, policy: str, capacity_factor: float, K: int, T: int,
                rho=None, num_ranks: int = 1) -> np.ndarray:
    """C_i^keep under the capacity policy ("Section 10.3"; Eq. 21, 23, 25).

    * ``none``: every request is kept.
    * ``per_expert``: C_keep = min(C_req, b).
    * ``rank_wide``: each destination q walks its local experts in ascending
      expert index (local-expert-major order) and admits routes cumulatively
      until its budget B is used up: keep_e = min(C_e^req, B - admitted so far).
    """
    C_req = np.asarray(C_req, np.int64)
    N = len(C_req)
    lim = capacity_limits(policy, capacity_factor, K, T, N, num_ranks)
    if lim is None:
        return C_req.copy()
    if policy == "per_expert":
        return np.minimum(C_req, lim)
    keep = np.zeros(N, np.int64)
    used = np.zeros(num_ranks, np.int64)
    for e in range(N):                      # ascending e is local-expert-major within each rank
        q = int(rho[e])
        keep[e] = min(int(C_req[e]), lim - int(used[q]))
        used[q] += keep[e]
    return keep


def pack_routes(idx, C_keep, N: int):
    """Keep flags, packed positions and the packed source map ("Section 10.3", Eq. 26).

    Readings: with one source, the kept routes of expert e are the first
    C_e^keep of its requests in token order (the prefix within each
    source/expert split).  Packed rows are ordered by expert, then by token
    (segments packed at the front, offsets o_e = sum_{i<e} M_i, M_i = C_i^keep).
    Returns (route_pos [T, K], -1 where dropped; perm_src [sum C_keep]; offsets [N+1]).
    """
    idx = np.asarray(idx)
    T, K = idx.shape
    C_keep = np.asarray(C_keep, np.int64)
    offsets = np.zeros(N + 1, np.int64)
    offsets[1:] = np.cumsum(C_keep)
    route_pos = np.full((T, K), -1, np.int64)
    perm_src = np.zeros(int(offsets[N]), np.int64)
    seen = np.zeros(N, np.int64)
    for t in range(T):                      # token order decides which requests are kept
        for k in range(K):
            e = int(idx[t, k])
            rank = int(seen[e])
            seen[e] += 1
            if rank < C_keep[e]:
                pos = int(offsets[e]) + rank
                route_pos[t, k] = pos
                perm_src[pos] = t
    return route_pos, perm_src, offsets


def drop_statistics(route_pos, r, C_req, C_keep, K: int, T: int) -> dict:
    """Drop diagnostics ("Section 10.3", Eq. 27 and the text after it).

    delta_route = sum D / (K T); tokens that lose at least one route; tokens
    that lose all K; the selected coefficient mass removed by dropping.
    """
    dropped = np.asarray(route_pos) < 0
    D = np.asarray(C_req) - np.asarray(C_keep)
    return {
        "delta_route": float(D.sum()) / float(K * T) if T > 0 else 0.0,
        "dropped_routes": int(D.sum()),
        "tokens_lost_any": int(dropped.any(axis=1).sum()),
        "tokens_lost_all": int(dropped.all(axis=1).sum()),
        "removed_weight": float(np.asarray(r)[dropped].sum()),
    }


# --------------------------------------------------------------------------- #
# Experts and the merge                                                        #
# --------------------------------------------------------------------------- #

def silu(a) -> np.ndarray:
    """SiLU(a) = a sigma(a)."""
    return f64(a) * sigmoid(a)


def swiglu(x, W_gate, W_up, W_down) -> np.ndarray:
    """E(x) = [SiLU(x W_g) (.) (x W_u)] W_d ("Section 20.1", Eq. 74), row-vector form.

    Storage: ``W_gate``/``W_up`` hold one row per intermediate unit ([m, d], so
    x W_g = x W_gate^T); ``W_down`` holds one row per output dimension ([d, m],
    so h W_d = h W_down^T).  No intermediate rounding.
    """
    x = f64(x)
    a = x @ f64(W_gate).T
    b = x @ f64(W_up).T
    return (silu(a) * b) @ f64(W_down).T


def merge_shared(parts: Sequence[Tuple]) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """W* of Eq. 75: concatenate gate and up columns, stack down rows ("Section 20.1").

    In the storage layout (gate/up one row per unit, down one column per unit)
    that is a row concatenation of gate/up and a column concatenation of down.
    """
    Wg = np.concatenate([f64(p[0]) for p in parts], axis=0)
    Wu = np.concatenate([f64(p[1]) for p in parts], axis=0)
    Wd = np.concatenate([f64(p[2]) for p in parts], axis=1)
    return Wg, Wu, Wd


def width_weighted_mean(r, s, d_r: int, d_s: int) -> float:
    """a_w = (d_r sum_i r_i + d_s s) / (K d_r + d_s) ("Section 21.1", Eq. 84)."""
    r = f64(r)
    K = r.shape[-1]
    return float((d_r * r.sum() + d_s * s) / (K * d_r + d_s))


def variance_ratio(r, s, d_r: int, d_s: int) -> float:
    """R_var = (d_r sum_i r_i^2 + d_s s^2) / (K d_r + d_s) ("Section 21.2", Eq. 85)."""
    r = f64(r)
    K = r.shape[-1]
    return float((d_r * (r ** 2).sum() + d_s * s * s) / (K * d_r + d_s))


def drop_totals(C_req_local, B: int, b) -> Tuple[int, int]:
    """D^rank = [sum_j C_j - B]_+ and D^expert = sum_j [C_j - b_j]_+ ("Section 10.4", Eq. 28)."""
    C = np.asarray(C_req_local, np.int64)
    b = np.asarray(b, np.int64)
    return max(int(C.sum()) - int(B), 0), int(np.maximum(C - b, 0).sum())


# --------------------------------------------------------------------------- #
# The whole layer                                                               #
# --------------------------------------------------------------------------- #

@dataclasses.dataclass
class Routing:
    logits: np.ndarray        # [T, N] the keys the selection used (float64 copy)
    topk_idx: np.ndarray      # [T, K]
    topk_w: np.ndarray        # [T, K] r = alpha * w
    counts_req: np.ndarray    # [N]
    counts_keep: np.ndarray   # [N]
    R_req: np.ndarray         # [M_E]
    R_keep: np.ndarray        # [M_E]
    offsets: np.ndarray       # [N + 1]
    route_pos: np.ndarray     # [T, K], -1 = dropped
    perm_src: np.ndarray      # [sum C_keep]
    drops: dict


def selection_keys(logits, selection_bias=None) -> np.ndarray:
    """a_t,i + b_i of Eq. 35: the key the selection ranks, with the persistent
    selection-only bias b ("Section 10.6", Eq. 35).  The bias moves the selection
    only; the mixture weights come from the unbiased logits.

    The key is formed in float32 (the precision of the device's logits), so the
    comparisons that decide the selection are the same on both sides.
    """
    z = np.asarray(logits)
    if selection_bias is None:
        return f64(z)
    return (z.astype(np.float32) + np.asarray(selection_bias, np.float32)[None, :]).astype(F64)


def route(logits, cfg, rho=None, selection_bias=None) -> Routing:
    """Steps from the logits to the packed layout, for a whole batch.

    ``cfg`` needs N, K, T, score, norm, alpha, cap_policy, capacity_factor,
    num_ranks (and norm_p for the L_p rule).  ``rho`` defaults to i mod num_ranks.  ``selection_bias`` is the
    optional Eq. 35 bias b (selection only).
    """
    z = f64(logits)
    T, N = z.shape
    K = cfg.K
    if rho is None:
        rho = [i % cfg.num_ranks for i in range(N)]
    idx = select_topk(selection_keys(logits, selection_bias), K)
    r = cfg.alpha * selected_weights(z, idx, cfg.score, cfg.norm, getattr(cfg, "norm_p", 2.0))
    C_req = requested_counts(idx, N)
    C_keep = kept_counts(C_req, cfg.cap_policy, cfg.capacity_factor, K, T, rho, cfg.num_ranks)
    route_pos, perm_src, offsets = pack_routes(idx, C_keep, N)
    return Routing(
        logits=z, topk_idx=idx, topk_w=r, counts_req=C_req, counts_keep=C_keep,
        R_req=destination_totals(C_req, rho, cfg.num_ranks),
        R_keep=destination_totals(C_keep, rho, cfg.num_ranks),
        offsets=offsets, route_pos=route_pos, perm_src=perm_src,
        drops=drop_statistics(route_pos, r, C_req, C_keep, K, T))


def moe_outputs_for_tokens(tokens, x_rows, routing: Routing, expert_weights: Callable,
                           shared_weights: Optional[Tuple], s_rows) -> np.ndarray:
    """y_t = sum_{k kept} r_t,k f_{S_t,k}(x_t) + s(x_t) g(x_t) ("Section 21", Eq. 80).

    Computes y for the listed tokens only.  ``expert_weights(e)`` returns
    (W_gate, W_up, W_down) of routed expert e; ``shared_weights`` is the merged
    shared expert or None.  Reading: a dropped route contributes nothing and
    the kept coefficients are not renormalised (the pages measure the weight
    removed by dropping), so a fully dropped token keeps only s(x) g(x).
    """
    tokens = np.asarray(tokens, np.int64)
    x_rows = f64(x_rows)
    d = x_rows.shape[1]
    y = np.zeros((len(tokens), d), F64)
    idx = routing.topk_idx[tokens]
    kept = routing.route_pos[tokens] >= 0
    r = routing.topk_w[tokens]
    for e in np.unique(idx[kept]):
        Wg, Wu, Wd = expert_weights(int(e))
        rows, slots = np.nonzero((idx == e) & kept)
        f = swiglu(x_rows[rows], Wg, Wu, Wd)
        y[rows] += r[rows, slots][:, None] * f
    if shared_weights is not None:
        g = swiglu(x_rows, *shared_weights)
        y += f64(s_rows)[:, None] * g
    return y


def moe_forward(cfg, inputs: dict, logits=None):
    """The full layer forward for a whole batch: returns (y [T, d], Routing, s [T]).

    ``inputs`` holds the tensors of the workload layout (x, W_router,
    router_bias, shared_gate_w, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
    and optionally the Eq. 35 selection_bias).
    ``logits``, when given, replaces the router projection (used to run the
    selection on exactly the keys another implementation computed).
    """
    x = inputs["x"]
    z = router_logits(x, inputs["W_router"], inputs.get("router_bias")) if logits is None else logits
    routing = route(z, cfg, selection_bias=inputs.get("selection_bias"))
    s = shared_coefficient(x, cfg.shared_mode, cfg.shared_gain, inputs.get("shared_gate_w"))
    Wg, Wu, Wd = inputs["W_gate"], inputs["W_up"], inputs["W_down"]
    shared = None
    if cfg.d_shared > 0 and cfg.shared_mode != "none":
        shared = (inputs["Ws_gate"], inputs["Ws_up"], inputs["Ws_down"])
    T = z.shape[0]
    y = moe_outputs_for_tokens(np.arange(T), x, routing, lambda e: (Wg[e], Wu[e], Wd[e]),
                               shared, s)
    return y, routing, s


# --------------------------------------------------------------------------- #
# Load-balancing statistics and the bias controller                           #
# --------------------------------------------------------------------------- #

def normalized_scores(z, score: str) -> np.ndarray:
    """p_t,i: router scores normalised across the N experts of each token.

    Softmax scores are already normalised; sigmoid scores are divided by their
    sum over the experts ("Section 10.7.1": for sigmoid routing the scores the
    loss uses are normalised across experts).
    """
    if score == "softmax":
        return softmax_all(z)
    q = sigmoid(z)
    return q / q.sum(axis=1, keepdims=True)


def lbl_statistics(p, idx, N: int):
    """f_i = C_i^req / (K T), P_i = mean_t p_t,i and L = N sum_i f_i P_i
    ("Section 10.5", Eq. 30; Eq. 38)."""
    p = f64(p)
    idx = np.asarray(idx)
    T, K = idx.shape
    C = requested_counts(idx, N).astype(F64)
    f = C / (K * T)
    P = p.mean(axis=0)
    return f, P, float(N * (f * P).sum())


def max_mean_imbalance(x) -> float:
    """I_max(x) = n ||x||_inf / ||x||_1 for a nonzero load vector ("Section 10.2", Eq. 22)."""
    x = f64(x)
    return float(len(x) * x.max() / x.sum())


def entropy_deficit(x) -> float:
    """I_H(x) = 1 - H(pi) / log n with pi = x / sum x ("Section 10.2").  With one expert
    (n = 1) the ratio is 0/0; a single expert cannot be imbalanced, so the deficit is 0."""
    x = f64(x)
    if len(x) < 2:
        return 0.0
    pi = x / x.sum()
    nz = pi[pi > 0]
    return float(1.0 + (nz * np.log(nz)).sum() / np.log(len(x)))


def coefficient_of_variation(x) -> float:
    """Standard deviation over mean of a load vector ("Section 10.2")."""
    x = f64(x)
    return float(x.std() / x.mean())


def never_selected(x) -> int:
    """Experts with zero load ("Section 10.2": never-selected experts)."""
    return int((np.asarray(x) == 0).sum())


def bias_update(bias, counts, gamma: float) -> np.ndarray:
    """b_i <- b_i + gamma sign(mean(C) - C_i) ("Section 10.6", Eq. 36-37).

    Computed in float32, the precision of the stored bias.
    """
    C = f64(counts)
    step = np.sign(C.mean() - C).astype(np.float32)
    return np.asarray(bias, np.float32) + np.float32(gamma) * step
