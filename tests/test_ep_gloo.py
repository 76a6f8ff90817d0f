"""Expert parallelism across two ranks on the CPU (gloo), against the oracle.

Each rank holds half of a batch and the experts rho(e) = e mod 2 maps to it.  It routes its
own tokens, all-gathers the requested split counts, derives the keep matrix and its routes'
destination rows with the library's host entries (Section 10.3, Eq. 23 and 26), sends its
kept rows to the experts' ranks, runs its local experts on what it received, gets the outputs
back and merges them (Eq. 80).  Checked against the oracle run on the two halves
concatenated in rank order (one batch, rank-wide capacity over the same two ranks):
- every rank derives the same keep matrix, and its column sums are the oracle's kept counts;
- each route is kept exactly when the oracle keeps it, at the row the oracle's packed
  layout gives it within its expert's rank;
- the merged outputs equal the oracle's y.
The expert arithmetic in the ranks is the oracle's SwiGLU (this is a test of the planning
and the exchange; the library's kernels need a GPU).
"""
import os
import socket

import numpy as np
import pytest
import torch

from tests.conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class Spec:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def _spec(T, cap):
    return Spec(T=T, d_model=32, N=8, K=2, d_expert=16, d_shared=16, score="softmax", norm="l1",
                alpha=2.0, cap_policy=cap, capacity_factor=0.7, num_ranks=2, shared_mode="const",
                shared_gain=1.0, norm_p=2.0)


def _inputs(T_total):
    g = torch.Generator().manual_seed(5)
    d, N, dr, ds = 32, 8, 16, 16
    r = lambda *s, sc: torch.randn(*s, generator=g, dtype=torch.float64) * sc
    # a per-expert logit bias skews the load so that the rank-wide budget drops routes
    return {"x": r(T_total, d, sc=1.0), "W_router": r(N, d, sc=0.3),
            "router_bias": torch.linspace(1.5, -1.5, N, dtype=torch.float64),
            "W_gate": r(N, dr, d, sc=d ** -0.5), "W_up": r(N, dr, d, sc=d ** -0.5),
            "W_down": r(N, d, dr, sc=dr ** -0.5), "Ws_gate": r(ds, d, sc=d ** -0.5),
            "Ws_up": r(ds, d, sc=d ** -0.5), "Ws_down": r(d, ds, sc=ds ** -0.5)}


def _worker(rank, world, port, cap, T_half, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from routing_shared_expert_gb300 import ep
        inp = _inputs(world * T_half)
        sl = slice(rank * T_half, (rank + 1) * T_half)
        x = inp["x"][sl]
        spec = _spec(T_half, "none")
        z = O.router_logits(x.numpy(), inp["W_router"].numpy(), inp["router_bias"].numpy())
        rt = O.route(z, spec)                       # this rank's own routing, no capacity
        topk = torch.as_tensor(rt.topk_idx, dtype=torch.int32)
        counts = torch.as_tensor(rt.counts_req, dtype=torch.int32)
        rho = [e % world for e in range(spec.N)]
        mine = [e for e in range(spec.N) if rho[e] == rank]

        def expert_fn(rows, off):
            out = torch.zeros_like(rows)
            for j, e in enumerate(mine):
                a, b = int(off[j]), int(off[j + 1])
                if b > a:
                    out[a:b] = torch.as_tensor(O.swiglu(rows[a:b].numpy(), inp["W_gate"][e].numpy(),
                                                        inp["W_up"][e].numpy(), inp["W_down"][e].numpy()))
            return out

        g = O.swiglu(x.numpy(), inp["Ws_gate"].numpy(), inp["Ws_up"].numpy(), inp["Ws_down"].numpy())

        def merge_fn(route_out, kept):
            f = route_out.numpy().reshape(T_half, spec.K, -1)
            r = rt.topk_w * kept.numpy()
            return torch.as_tensor((r[:, :, None] * f).sum(1) + 1.0 * g)

        y, plan = ep.ep_layer_forward(x, topk, rho, spec.K, expert_fn, merge_fn, counts, cap, 0.7)
        q.put((rank, {"y": y.numpy(), "keep": plan.keep.numpy(), "dst": plan.dst_row.numpy(),
                      "R_keep": plan.R_keep.numpy(), "R_req": plan.R_req.numpy()}))
    except Exception as e:  # report to the parent instead of hanging it
        import traceback
        q.put((rank, traceback.format_exc()))
    finally:
        dist.destroy_process_group()


def _run(cap, T_half=160, world=2):
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cap, T_half, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, res = q.get(timeout=240)
        assert not isinstance(res, str), res
        got[rank] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("cap", ["rank_wide", "none"])
def test_two_ranks_match_the_oracle_on_the_concatenated_batch(cap):
    import oracle as O
    T_half, world = 160, 2
    got = _run(cap, T_half, world)
    inp = _inputs(world * T_half)
    spec = _spec(world * T_half, cap)
    y_ref, rt, _ = O.moe_forward(spec, {k: v.numpy() for k, v in inp.items()})
    # every rank derives the same keep matrix; its column sums are the oracle's kept counts
    keep = got[0]["keep"]
    assert np.array_equal(keep, got[1]["keep"])
    assert np.array_equal(keep.sum(0), rt.counts_keep)
    assert np.array_equal(got[0]["R_keep"], rt.R_keep) and np.array_equal(got[0]["R_req"], rt.R_req)
    if cap == "rank_wide":
        assert rt.drops["dropped_routes"] > 0
    # each route kept exactly when the oracle keeps it, at its row within its expert's rank
    rho = np.arange(spec.N) % world
    off_in_rank = np.zeros(spec.N, np.int64)
    for qd in range(world):
        run = 0
        for e in range(spec.N):
            if rho[e] == qd:
                off_in_rank[e] = run
                run += rt.counts_keep[e]
    dst = np.concatenate([got[r]["dst"] for r in range(world)])
    pos = rt.route_pos
    e_of = rt.topk_idx
    want = np.where(pos >= 0, off_in_rank[e_of] + pos - rt.offsets[e_of], -1)
    assert np.array_equal(dst, want)
    # the merged outputs
    y = np.concatenate([got[r]["y"] for r in range(world)])
    assert np.abs(y - y_ref).max() <= 1e-12 * np.abs(y_ref).max()
