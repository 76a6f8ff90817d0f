"""Expert-parallel capacity agreement (Section 10.3, Eq. 23 and Eq. 26): the library's host
entries on hand-worked keep matrices (CPU only)."""
import ctypes

import pytest
import torch

from tests.conftest import ensure_built


@pytest.fixture(scope="module")
def nat():
    ensure_built()
    from routing_shared_expert_gb300 import _native
    return _native


def _keep(nat, counts, rho, K, policy, c):
    M, N = len(counts), len(counts[0])
    cnt = torch.tensor(counts, dtype=torch.int32)
    keep = torch.empty((M, N), dtype=torch.int32)
    off = torch.empty((M, N), dtype=torch.int32)
    rq = torch.empty(M, dtype=torch.int32)
    rk = torch.empty(M, dtype=torch.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = nat.library().moe_ep_keep_matrix_host(M, N, K, (ctypes.c_int32 * N)(*rho), policy, c, p(cnt),
                                               p(keep), p(off), p(rq), p(rk))
    return st, keep.tolist(), off.tolist(), rq.tolist(), rk.tolist()


def test_two_sources_by_hand(nat):
    """Two sources, four experts, rho = (0, 0, 1, 1), top-1, c = 1: twelve tokens, so each
    destination's budget is ceil(1 * 1 * 12 / 2) = 6.  Destination 0 admits (e0, s0) = 4,
    (e0, s1) = 2, then nothing of (e1, s1) = 2; destination 1 keeps all four of its rows."""
    st, keep, off, rq, rk = _keep(nat, [[4, 0, 1, 1], [2, 2, 1, 1]], [0, 0, 1, 1], 1, 2, 1.0)
    assert st == 0
    assert keep == [[4, 0, 1, 1], [2, 0, 1, 1]]
    # rows of destination 0: e0 from s0 at 0-3, e0 from s1 at 4-5; destination 1: e2 s0, e2
    # s1, e3 s0, e3 s1 at 0, 1, 2, 3
    assert off == [[0, 6, 0, 2], [4, 6, 1, 3]]
    assert rq == [8, 4] and rk == [6, 4]
    # without capacity every request is kept
    st, keep, off, rq, rk = _keep(nat, [[4, 0, 1, 1], [2, 2, 1, 1]], [0, 0, 1, 1], 1, 0, 1.0)
    assert keep == [[4, 0, 1, 1], [2, 2, 1, 1]] and rk == rq == [8, 4]
    assert off == [[0, 6, 0, 2], [4, 6, 1, 3]]


def test_placement_keeps_a_prefix_of_each_split(nat):
    """Source 1 of the case above: its tokens request experts (1, 0, 1, 0, 2, 3) in token order;
    keep[1] = (2, 0, 1, 1): both e0 routes kept at rows 4, 5, both e1 routes dropped."""
    _, keep, off, _, _ = _keep(nat, [[4, 0, 1, 1], [2, 2, 1, 1]], [0, 0, 1, 1], 1, 2, 1.0)
    idx = torch.tensor([[1], [0], [1], [0], [2], [3]], dtype=torch.int32)
    keep_t = torch.tensor(keep, dtype=torch.int32)
    off_t = torch.tensor(off, dtype=torch.int32)
    dst = torch.empty((6, 1), dtype=torch.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert nat.library().moe_ep_place_host(2, 1, 6, 4, 1, p(idx), p(keep_t), p(off_t), p(dst)) == 0
    assert dst.reshape(-1).tolist() == [-1, 4, -1, 5, 1, 3]


def test_bad_arguments_rejected(nat):
    st, *_ = _keep(nat, [[1, 1], [1, 1]], [0, 2], 1, 2, 1.0)     # rho out of range
    assert st == -1
    st, *_ = _keep(nat, [[1, 1], [1, 1]], [0, 1], 1, 1, 1.0)     # per-expert capacity
    assert st == -2
    st, *_ = _keep(nat, [[1, 1], [1, 1]], [0, 1], 1, 2, 0.0)     # c must be positive
    assert st == -1
    # a source rank outside [0, M) is rejected before any array is read
    idx = torch.zeros((2, 1), dtype=torch.int32)
    keep = torch.zeros((2, 2), dtype=torch.int32)
    dst = torch.empty((2, 1), dtype=torch.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert nat.library().moe_ep_place_host(2, 2, 2, 2, 1, p(idx), p(keep), p(keep), p(dst)) == -1
    assert nat.library().moe_ep_place_host(2, -1, 2, 2, 1, p(idx), p(keep), p(keep), p(dst)) == -1


def test_send_positions_and_receive_rows_by_hand(nat):
    """The case above.  Source 1 sends, to destination 0, its e0 rows (keep 2) and, to
    destination 1, its e2 and e3 rows: routes (1, 0, 1, 0, 2, 3) land at send rows
    (-, 0, -, 1, 2, 3).  Destination 0 receives source 0's four e0 rows, then source 1's two:
    packed rows 0-5 in order; destination 1 receives source 0's e2, e3 (packed rows 0, 2) then
    source 1's e2, e3 (rows 1, 3)."""
    _, keep, off, _, _ = _keep(nat, [[4, 0, 1, 1], [2, 2, 1, 1]], [0, 0, 1, 1], 1, 2, 1.0)
    rho = (ctypes.c_int32 * 4)(0, 0, 1, 1)
    keep_t = torch.tensor(keep, dtype=torch.int32)
    off_t = torch.tensor(off, dtype=torch.int32)
    idx = torch.tensor([[1], [0], [1], [0], [2], [3]], dtype=torch.int32)
    dst = torch.tensor([[-1], [4], [-1], [5], [1], [3]], dtype=torch.int32)
    pos = torch.empty((6, 1), dtype=torch.int32)
    cnt = torch.empty(2, dtype=torch.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    lib = nat.library()
    assert lib.moe_ep_send_pos_host(2, 1, 6, 4, 1, rho, p(idx), p(keep_t), p(off_t), p(dst), p(pos),
                                    p(cnt)) == 0
    assert pos.reshape(-1).tolist() == [-1, 0, -1, 1, 2, 3] and cnt.tolist() == [2, 2]
    for q, want in ((0, [0, 1, 2, 3, 4, 5]), (1, [0, 2, 1, 3])):
        rr = torch.empty(len(want), dtype=torch.int32)
        assert lib.moe_ep_recv_rows_host(2, q, 4, rho, p(keep_t), p(off_t), p(rr), len(want)) == 0
        assert rr.tolist() == want
    # a receive buffer one row short is rejected
    rr = torch.empty(3, dtype=torch.int32)
    assert lib.moe_ep_recv_rows_host(2, 1, 4, rho, p(keep_t), p(off_t), p(rr), 3) == -1


def test_rows_copy_host(nat):
    """dst[dst_index[i]] = src[src_index[i]] (or src[i / src_div]); negative destinations skip,
    negative sources zero the row when asked; indices past the buffers are rejected."""
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    lib = nat.library()
    src = torch.arange(3 * 4, dtype=torch.float32).reshape(3, 4)          # 16-byte rows
    dst = torch.full((6, 4), -1.0)
    # route -> token: 6 routes of K = 2 over 3 tokens, scattered to rows 5..0, route 2 dropped
    di = torch.tensor([5, 4, -1, 2, 1, 0], dtype=torch.int32)
    assert lib.moe_rows_copy_host(p(src), 3, None, 2, p(dst), 6, p(di), 6, 16, 0) == 0
    want = torch.full((6, 4), -1.0)
    for i, t in enumerate(di.tolist()):
        if t >= 0:
            want[t] = src[i // 2]
    assert torch.equal(dst, want)
    # gather with a missing source, zeroed
    si = torch.tensor([2, -1, 0], dtype=torch.int32)
    out = torch.full((3, 4), 7.0)
    assert lib.moe_rows_copy_host(p(src), 3, p(si), 1, p(out), 3, None, 3, 16, 1) == 0
    assert torch.equal(out, torch.stack([src[2], torch.zeros(4), src[0]]))
    # out of range, a row size that is not a multiple of 16 bytes, and a bad divisor
    bad = torch.tensor([3], dtype=torch.int32)
    assert lib.moe_rows_copy_host(p(src), 3, p(bad), 1, p(out), 3, None, 1, 16, 0) == -1
    assert lib.moe_rows_copy_host(p(src), 3, None, 1, p(out), 3, None, 1, 12, 0) == -2
    assert lib.moe_rows_copy_host(p(src), 3, None, 0, p(out), 3, None, 1, 16, 0) == -1
