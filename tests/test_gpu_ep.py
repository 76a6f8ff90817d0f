"""The expert-parallel planning entries on the device (GB300), against their host twins.

moe_ep_keep_matrix derives the keep matrix from all-gathered counts on the device (the
token total recovered from the counts), and moe_ep_place gives each route of a source its
destination row from the stable ranks of a capacity-free moe_permute of that source's
batch.  Both must equal the host entries (which the two-rank gloo test checks against the
oracle) bit for bit, for several source counts, with and without the rank-wide budget.
The exchange kernels (send positions, receive rows, indexed row copies) are checked by
running the dispatch and the return of M sources on one GPU, the all-to-all itself replaced
by slicing the send buffers.
"""
import ctypes

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
    for k in ("keep", "recv_off", "R_req", "R_keep", "dst_row", "send_pos"):
        assert torch.equal(getattr(dev, k).cpu(), getattr(host, k)), k
    assert moe.moe_read_status(ws) == 0
    if cap == "rank_wide" and M > 1:
        assert int(host.keep.sum()) < int(counts.sum())   # the budget dropped some routes


def _route_source(spec, seed):
    cfg = moe.config_from_spec(spec)
    inp = make_inputs(spec, "cuda", seed=seed)
    ws = moe.alloc_workspace(cfg)
    T, K, N = spec.T, spec.K, spec.N
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["W_router"], None, None, None, idx, w, None, None, ws)
    cnt = torch.empty(N, dtype=torch.int32, device="cuda")
    ck = torch.empty(N, dtype=torch.int32, device="cuda")
    off = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    rpos = torch.empty((T, K), dtype=torch.int32, device="cuda")
    psrc = torch.empty(T * K, dtype=torch.int32, device="cuda")
    moe.moe_permute(cfg, None, idx, cnt, ck, off, rpos, psrc, None, None, None, None, ws)
    return inp["x"], idx, cnt, off, rpos, ws


@pytest.mark.parametrize("M", [1, 3])
def test_device_exchange_of_m_sources(M):
    """Dispatch: every kept route's x row reaches row dst_row of destination rho(e)'s packed
    buffer; return: every route gets back its row of the destination's outputs (here 2 x the
    row), dropped routes zero.  All row movement by the library's kernels."""
    spec = CONFIGS["dsv3"].replace(T=300, d_model=256, N=32, K=4, d_expert=128, d_shared=128)
    N, K, T, d = spec.N, spec.K, spec.T, spec.d_model
    rho = [e % M for e in range(N)]
    src = [_route_source(spec, seed=11 + s) for s in range(M)]
    counts = torch.stack([c for (_, _, c, _, _, _) in src])
    plans = [ep.make_plan(counts, src[s][1], s, K, rho, "rank_wide", 0.6, route_pos=src[s][4],
                          offsets=src[s][3], workspace=src[s][5]) for s in range(M)]
    split = plans[0].send_counts()                      # [source, destination] rows
    sends = []
    for s in range(M):
        buf = torch.empty((int(split[s].sum()), d), dtype=torch.bfloat16, device="cuda")
        ep.rows_copy(src[s][0], buf, T * K, src_div=K, dst_index=plans[s].send_pos,
                     workspace=src[s][5])
        sends.append(buf)
    start = torch.cat([torch.zeros((M, 1), dtype=torch.int64), split.cumsum(1)], 1)
    packed = []
    for q in range(M):
        # the all-to-all: destination q receives source s's block for q, sources in order
        recv = torch.cat([sends[s][int(start[s, q]):int(start[s, q + 1])] for s in range(M)])
        rr = ep.recv_rows(plans[q], workspace=src[q][5])
        rows = torch.zeros((int(plans[q].R_keep[q]), d), dtype=torch.bfloat16, device="cuda")
        ep.rows_copy(recv, rows, recv.shape[0], dst_index=rr, workspace=src[q][5])
        packed.append((rows, rr, recv.shape[0]))
    torch.cuda.synchronize()
    # every kept route's row sits at its destination row
    for s in range(M):
        x, idx = src[s][0], src[s][1]
        dst = plans[s].dst_row
        kept = dst >= 0
        q_of = torch.tensor(rho, device="cuda")[idx.long()]
        for q in range(M):
            sel = kept & (q_of == q)
            t = torch.nonzero(sel)[:, 0]
            assert torch.equal(packed[q][0][dst[sel].long()], x[t])
        if M > 1:
            assert int((~kept).sum()) > 0   # the budget dropped some routes
    # the return path: each destination's outputs (2 x its rows) go back to the sources
    backs = {}
    for q in range(M):
        rows, rr, n = packed[q]
        f = rows * 2
        send_back = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
        ep.rows_copy(f, send_back, n, src_index=rr, workspace=src[q][5])
        backs[q] = send_back
    rstart = torch.cat([torch.zeros((1, M), dtype=torch.int64), split.cumsum(0)], 0)
    for s in range(M):
        back = torch.cat([backs[q][int(rstart[s, q]):int(rstart[s + 1, q])] for q in range(M)])
        out = torch.full((T * K, d), 5.0, dtype=torch.bfloat16, device="cuda")
        ep.rows_copy(back, out, T * K, src_index=plans[s].send_pos, zero_missing=True,
                     workspace=src[s][5])
        torch.cuda.synchronize()
        kept = (plans[s].dst_row >= 0).reshape(-1)
        want = (src[s][0] * 2).repeat_interleave(K, 0)
        want[~kept] = 0
        assert torch.equal(out, want)
    for s in range(M):
        assert moe.moe_read_status(src[s][5]) == 0


def _ep_nccl_worker(port, q):
    """One NCCL rank: the expert-parallel forward with the library's kernels throughout."""
    import sys
    from tests.conftest import ROOT
    sys.path.insert(0, ROOT)
    try:
        import torch.distributed as dist
        torch.cuda.set_device(0)
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1)
        spec = CONFIGS["dsv3"].replace(T=600, d_model=256, N=32, K=4, d_expert=128,
                                       d_shared=128, cap_policy="rank_wide",
                                       capacity_factor=0.7, num_ranks=1)
        T, K, N, d = spec.T, spec.K, spec.N, spec.d_model
        inp = make_inputs(spec, "cuda")
        layer = moe.MoELayer(moe.config_from_spec(spec), inp, "cuda")
        y_ref = layer.forward(inp["x"], logits=False).clone()
        cfg, ws, x = layer.cfg, layer.ws, inp["x"]
        i32 = dict(dtype=torch.int32, device="cuda")
        idx, cnt, ck, off = (torch.empty((T, K), **i32), torch.empty(N, **i32),
                             torch.empty(N, **i32), torch.empty(N + 1, **i32))
        rpos, psrc = torch.empty((T, K), **i32), torch.empty(T * K, **i32)
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        sc = torch.empty(T, dtype=torch.float32, device="cuda")
        moe.moe_route(cfg, x, inp["W_router"], None, None, None, idx, w, sc, None, ws)
        moe.moe_permute(moe.copy_config(cfg, cap_policy=0), None, idx, cnt, ck, off, rpos, psrc,
                        None, None, None, None, ws)
        g = torch.empty((T, d), dtype=torch.float16, device="cuda")
        moe.moe_shared_mlp(cfg, x, inp["Ws_gate"], inp["Ws_up"], layer.down["Ws_down"], g, ws)

        def expert_fn(rows, local_off):
            buf = torch.zeros((T * K, d), dtype=torch.bfloat16, device="cuda")
            buf[:rows.shape[0]] = rows
            f = torch.zeros((T * K, d), dtype=torch.float16, device="cuda")
            moe.moe_grouped_swiglu(cfg, buf, local_off.to(torch.int32).cuda(), None,
                                   inp["W_gate"], inp["W_up"], layer.down["W_down"], f, ws)
            return f[:rows.shape[0]]

        def merge_fn(route_out, kept):
            rp = torch.where(kept, torch.arange(T * K, **i32).view(T, K), -1).contiguous()
            y = torch.empty((T, d), dtype=torch.float32, device="cuda")
            moe.moe_combine(cfg, route_out, rp, w, g, sc, y)
            return y

        y, plan = ep.ep_layer_forward(x, idx, [0] * N, K, expert_fn, merge_fn, cnt, "rank_wide",
                                      0.7, route_pos=rpos, offsets=off, workspace=ws)
        torch.cuda.synchronize()
        dropped = int((plan.dst_row < 0).sum())
        q.put(("ok", bool(torch.equal(y, y_ref)), float((y - y_ref).abs().max()), dropped,
               moe.moe_read_status(ws)))
        dist.destroy_process_group()
    except Exception:
        import traceback
        q.put(("error", traceback.format_exc()))


def test_expert_parallel_forward_on_one_nccl_rank_equals_the_fused_layer():
    """ep_layer_forward over NCCL with one rank and the library's kernels for every step
    (router, capacity-free permutation, keep matrix, send and receive layouts, row copies,
    grouped experts, shared expert, combine) gives the fused layer's y under the same
    rank-wide budget bit for bit: the same kept rows in the same packed order."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_ep_nccl_worker, args=(port, q))
    p.start()
    res = q.get(timeout=300)
    p.join(timeout=60)
    assert res[0] == "ok", res[1]
    _, equal, err, dropped, status = res
    assert status == 0
    assert dropped > 0             # the budget is binding
    assert equal, f"max |y_ep - y_layer| = {err}"
    assert p.exitcode == 0


def test_device_rows_copy_and_send_pos_bounds():
    """An index past a buffer records MOE_ERR_DEVICE_BOUNDS in the workspace and skips that
    row (the others are copied); an expert id out of range gets send position -1 with the
    same status."""
    from routing_shared_expert_gb300 import _native as nat
    spec = CONFIGS["olmo"].replace(T=64, d_model=128, N=8, K=2, d_expert=128, d_shared=128)
    ws = moe.alloc_workspace(moe.config_from_spec(spec))
    src = torch.arange(4 * 8, dtype=torch.float32, device="cuda").reshape(4, 8)
    dst = torch.full((4, 8), -1.0, device="cuda")
    di = torch.tensor([3, 9, 1, 0], dtype=torch.int32, device="cuda")   # 9 is past dst
    ep.rows_copy(src, dst, 4, dst_index=di, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == -6  # MOE_ERR_DEVICE_BOUNDS
    want = torch.full((4, 8), -1.0, device="cuda")
    want[3], want[1], want[0] = src[0], src[2], src[3]
    assert torch.equal(dst, want)
    assert moe.moe_read_status(ws) == 0                                 # read clears it
    # send positions with one expert id out of range
    rho = [0, 1] * 4
    keep = torch.tensor([[2, 1, 1, 0, 0, 0, 0, 0], [0] * 8], dtype=torch.int32, device="cuda")
    off = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    idx = torch.tensor([[0, 1], [0, 12]], dtype=torch.int32, device="cuda")
    dst_row = torch.tensor([[0, 0], [1, -1]], dtype=torch.int32, device="cuda")
    pos = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    cnt = torch.empty(2, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = nat.library().moe_ep_send_pos(2, 0, 2, 8, 2, (ctypes.c_int32 * 8)(*rho), p(idx), p(keep),
                                       p(off), p(dst_row), p(pos), p(cnt), p(ws), ws.numel(),
                                       nat._stream(None))
    assert st == 0
    torch.cuda.synchronize()
    # experts of rank 0: 0, 2 (keep 2, 1) -> send rows 0-2; rank 1: 1 (keep 1) -> row 3
    assert pos.tolist() == [[0, 3], [1, -1]] and cnt.tolist() == [3, 1]
    assert moe.moe_read_status(ws) == -6  # MOE_ERR_DEVICE_BOUNDS
