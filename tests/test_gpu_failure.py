"""Device-detected failures reach the caller as status codes, without a GPU fault (GB300).

- A bounded wait that runs out: moe_check_wait_bound makes one CTA wait, with a short
  limit, on a barrier that nothing arrives on, through the same bounded wait every
  tensor-core kernel uses.  The status word then holds MOE_ERR_TIMEOUT, the call has
  taken about the limit, and the next layer call on the same workspace runs normally.
- An expert id out of range in topk_idx: the permutation's own bounds checks report
  MOE_ERR_DEVICE_BOUNDS and treat those routes as dropped (position -1), counting only
  the valid ones; the workspace is usable again once the status is read.
"""
import time

import pytest
import torch

import routing_shared_expert_gb300 as moe
from tests.gpu_helpers import run_layer
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

TIMEOUT = -5
DEVICE_BOUNDS = -6
SPEC = CONFIGS["olmo"].replace(T=500, d_model=256, d_expert=128, d_shared=128, alpha=2.0)


def test_bounded_wait_runs_out_and_reports():
    inp = make_inputs(SPEC, "cuda")
    layer = run_layer(SPEC, inp)
    y0 = layer.out["y"].clone()
    assert layer.status() == 0
    limit_ns = 20_000_000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_check_wait_bound(layer.ws, limit_ns)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert moe.moe_read_status(layer.ws) == TIMEOUT
    assert limit_ns * 1e-9 <= dt < 2.0, f"wait gave up after {dt:.3f} s"
    assert moe.moe_read_status(layer.ws) == 0     # read clears it
    # the context and the workspace are usable: the same call gives the same result
    y1 = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y1, y0)


def test_expert_id_out_of_range_is_reported_and_dropped():
    inp = make_inputs(SPEC, "cuda")
    layer = run_layer(SPEC, inp)
    o, c = layer.out, layer.cfg
    T, K, N, d = SPEC.T, SPEC.K, SPEC.N, SPEC.d_model
    idx = o["topk_idx"].clone()
    bad = [(3, 0, N), (17, 1, -1), (400, 0, N + 5)]
    for t, k, e in bad:
        idx[t, k] = e
    counts_req = torch.zeros(N, dtype=torch.int32, device="cuda")
    counts_keep = torch.zeros(N, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    route_pos = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    perm_src = torch.zeros(T * K, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((T * K, d), dtype=SPEC.torch_dtype, device="cuda")
    moe.moe_permute(c, inp["x"], idx, counts_req, counts_keep, offsets, route_pos, perm_src, x_perm,
                    None, None, None, layer.ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(layer.ws) == DEVICE_BOUNDS
    for t, k, _ in bad:
        assert int(route_pos[t, k]) == -1
    valid = (idx >= 0) & (idx < N)
    assert int(counts_req.sum()) == int(valid.sum()) == T * K - len(bad)
    ref = torch.bincount(idx[valid].long(), minlength=N).to(torch.int32)
    assert torch.equal(counts_req, ref)
    # every valid route got its packed row, and the rows hold the right tokens
    rows = route_pos[valid].long()
    assert torch.equal(torch.sort(rows).values, torch.arange(int(valid.sum()), device="cuda"))
    toks = torch.arange(T, device="cuda")[:, None].expand(T, K)[valid]
    assert torch.equal(perm_src[rows].long(), toks)
    assert torch.equal(x_perm[rows], inp["x"][toks])
    # the workspace works again once the status is read
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
