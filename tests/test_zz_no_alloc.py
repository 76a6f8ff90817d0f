"""moe_permute_noalloc: the permutation step for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc and have no workspace to give: a serving
process whose device memory is planned and reserved at start-up, or a plugin
host that hands over only the inputs and outputs of each call.  For them the
library offers moe_permute_noalloc, whose scratch is a fixed array built into
the library.  This test calls it through the C ABI twice in a row, on two
different layers, and checks every output against the regular moe_permute (which
takes a workspace): counts, capacity decisions, offsets, positions, the source
map and the gathered rows must agree bit for bit.  The second call also shows
that whatever the first call left in the shared array does not leak into the
next result.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from tests.conftest import ensure_built
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _route(moe, cfg, inp):
    T, K, N = cfg.T, cfg.K, cfg.N
    ws = moe.alloc_workspace(cfg)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["W_router"], inp["router_bias"], None, inp["shared_gate_w"],
                  idx, w, None, None, ws)
    return idx, ws


def _outputs(cfg, spec):
    T, K, N, d, M = cfg.T, cfg.K, cfg.N, cfg.d_model, cfg.num_ranks
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts_req=torch.full((N,), -7, **i32), counts_keep=torch.full((N,), -7, **i32),
                offsets=torch.full((N + 1,), -7, **i32), route_pos=torch.full((T, K), -7, **i32),
                perm_src=torch.full((T * K,), -7, **i32),
                x_perm=torch.zeros((T * K, d), dtype=spec.torch_dtype, device="cuda"),
                R_req=torch.full((M,), -7, **i32), R_keep=torch.full((M,), -7, **i32),
                drop_stats=torch.full((4,), -7, **i32))


def _compare(a, b):
    for k in ("counts_req", "counts_keep", "offsets", "route_pos", "R_req", "R_keep", "drop_stats"):
        assert torch.equal(a[k], b[k]), k
    kept = int(a["offsets"][-1])
    assert torch.equal(a["perm_src"][:kept], b["perm_src"][:kept])
    assert torch.equal(a["x_perm"][:kept], b["x_perm"][:kept])
    return kept


def test_permute_noalloc_matches_workspace_version_twice():
    ensure_built()
    import routing_shared_expert_gb300 as moe
    # call 1: capacity with drops (Mixtral recipe); call 2: a different layer without capacity
    specs = [CONFIGS["mixtral"].replace(T=1500, d_model=256, d_expert=128, capacity_factor=0.8),
             CONFIGS["dsv3"].replace(T=700, d_model=256, d_expert=128, d_shared=128)]
    for spec in specs:
        cfg = moe.config_from_spec(spec)
        inp = make_inputs(spec, "cuda")
        idx, ws = _route(moe, cfg, inp)
        ref = _outputs(cfg, spec)
        moe.moe_permute(cfg, inp["x"], idx, ref["counts_req"], ref["counts_keep"], ref["offsets"],
                        ref["route_pos"], ref["perm_src"], ref["x_perm"], ref["R_req"], ref["R_keep"],
                        ref["drop_stats"], ws)
        got = _outputs(cfg, spec)
        moe.moe_permute_noalloc(cfg, inp["x"], idx, got["counts_req"], got["counts_keep"],
                                got["offsets"], got["route_pos"], got["perm_src"], got["x_perm"],
                                got["R_req"], got["R_keep"], got["drop_stats"])
        torch.cuda.synchronize()
        kept = _compare(ref, got)
        assert kept > 0
        if spec.cap_policy != "none":
            assert int(got["drop_stats"][0]) > 0


def test_permute_noalloc_at_the_size_limit_and_without_row_copy():
    """ceil(T / 256) * N == 65536 exactly (T = 65536 at N = 256) uses the last histogram row of
    the static array; the result equals moe_permute's bit for bit.  A second call without
    x_perm (and without x: no rows copied, the expert GEMM can gather through perm_src)
    gives the same routing tables."""
    ensure_built()
    import routing_shared_expert_gb300 as moe
    spec = CONFIGS["dsv3"].replace(T=65536, d_model=64, d_expert=64, d_shared=64)
    cfg = moe.config_from_spec(spec)
    inp = make_inputs(spec, "cuda")
    idx, ws = _route(moe, cfg, inp)
    ref = _outputs(cfg, spec)
    moe.moe_permute(cfg, inp["x"], idx, ref["counts_req"], ref["counts_keep"], ref["offsets"],
                    ref["route_pos"], ref["perm_src"], ref["x_perm"], ref["R_req"], ref["R_keep"],
                    ref["drop_stats"], ws)
    got = _outputs(cfg, spec)
    moe.moe_permute_noalloc(cfg, inp["x"], idx, got["counts_req"], got["counts_keep"],
                            got["offsets"], got["route_pos"], got["perm_src"], got["x_perm"],
                            got["R_req"], got["R_keep"], got["drop_stats"])
    torch.cuda.synchronize()
    assert _compare(ref, got) == spec.T * spec.K
    bare = _outputs(cfg, spec)
    moe.moe_permute_noalloc(cfg, None, idx, bare["counts_req"], bare["counts_keep"],
                            bare["offsets"], bare["route_pos"], bare["perm_src"], None,
                            bare["R_req"], bare["R_keep"], bare["drop_stats"])
    torch.cuda.synchronize()
    bare["x_perm"] = ref["x_perm"]
    _compare(ref, bare)


def test_permute_noalloc_rejects_layers_beyond_its_scratch():
    ensure_built()
    import routing_shared_expert_gb300 as moe
    # one counting tile past the limit: ceil(T / 256) * 256 experts = 65792 > 65536
    spec = CONFIGS["dsv3"].replace(T=65536 + 1)
    cfg = moe.config_from_spec(spec)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_permute_noalloc(cfg, None, None, None, None, None, None, None, None, None, None,
                                None)
    assert e.value.status == -2
