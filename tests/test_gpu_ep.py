"""The expert-parallel planning entries on the device (GB300), against their host twins.

moe_ep_keep_matrix derives the keep matrix from all-gathered counts on the device (the
token total recovered from the counts), and moe_ep_place gives each route of a source its
destination row from the stable ranks of a capacity-free moe_permute of that source's
batch.  Both must equal the host entries (which the two-rank gloo test checks against the
oracle) bit for bit, for several source counts, with and without the rank-wide budget.
"""
import pytest
import torch

import routing_shared_expert_gb300 as moe
from routing_shared_expert_gb300 import ep
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("cap", ["rank_wide", "none"])
def test_device_plan_equals_host_plan(M, cap):
    spec = CONFIGS["dsv3"].replace(T=700, d_model=256, d_expert=128, d_shared=128)
    N, K = spec.N, spec.K
    rho = [e % M for e in range(N)]
    g = torch.Generator().manual_seed(3 + M)
    # requested counts of M sources (each row sums to K T_s for some T_s)
    counts = torch.zeros((M, N), dtype=torch.int32)
    for s in range(M):
        T_s = 300 + 50 * s
        idx = torch.stack([torch.randperm(N, generator=g)[:K] for _ in range(T_s)])
        counts[s] = torch.bincount(idx.reshape(-1), minlength=N).to(torch.int32)
    # source M - 1's batch on the device: its routing, and a capacity-free permutation
    cfg = moe.config_from_spec(spec)
    inp = make_inputs(spec, "cuda")
    ws = moe.alloc_workspace(cfg)
    T = spec.T
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["W_router"], None, None, None, idx, w, None, None, ws)
    cnt_src = torch.empty(N, dtype=torch.int32, device="cuda")
    ck = torch.empty(N, dtype=torch.int32, device="cuda")
    off = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    rpos = torch.empty((T, K), dtype=torch.int32, device="cuda")
    psrc = torch.empty(T * K, dtype=torch.int32, device="cuda")
    moe.moe_permute(cfg, None, idx, cnt_src, ck, off, rpos, psrc, None, None, None, None, ws)
    counts[M - 1] = cnt_src.cpu()   # the last source is the batch routed on the device
    host = ep.make_plan(counts, idx.cpu(), M - 1, K, rho, cap, 0.6)
    dev = ep.make_plan(counts.cuda(), idx, M - 1, K, rho, cap, 0.6, route_pos=rpos, offsets=off,
                       workspace=ws)
    torch.cuda.synchronize()
    for k in ("keep", "recv_off", "R_req", "R_keep", "dst_row"):
        assert torch.equal(getattr(dev, k).cpu(), getattr(host, k)), k
    assert moe.moe_read_status(ws) == 0
    if cap == "rank_wide" and M > 1:
        assert int(host.keep.sum()) < int(counts.sum())   # the budget dropped some routes
