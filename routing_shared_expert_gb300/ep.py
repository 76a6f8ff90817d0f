"""Expert parallelism across ranks: capacity agreement, dispatch and combine.

Section 10 "Routing, Capacity, and Load Balancing", Section 10.3 (Eq. 23 and Eq. 26,
Figure 41).  Each rank holds a batch of tokens and the experts rho maps to it.  Per forward:

1. each rank routes its own tokens and counts its requests per expert (C^req of its batch);
2. the ranks all-gather those N-length count vectors; each derives the same keep matrix and
   the destination row of each of its routes (``moe_ep_keep_matrix`` / ``moe_ep_place`` on
   CUDA tensors, their host twins on CPU tensors): destination q packs, per local expert in
   ascending index, the kept rows of source 0, then source 1, ...;
3. dispatch: each source lays its kept rows out in a send buffer (destinations in
   ascending rank, each in the destination's buffer order), one all-to-all moves them, and
   each destination scatters its receive buffer into its packed buffer
   (``moe_ep_send_pos``, ``moe_rows_copy``, ``moe_ep_recv_rows``);
4. each rank runs its local experts over its packed buffer (segments from the keep matrix);
5. combine: the expert outputs go back the same way (gather, reverse all-to-all, gather by
   send position), and each source merges them with its shared branch (Eq. 80; dropped
   routes add nothing).

This module plans and moves data with the library's entry points (on CUDA tensors the
device kernels, on CPU tensors their host twins); the routing, the expert GEMMs and the
merge are callables (on a GPU: the library's kernels).  The collectives are
``torch.distributed`` (NCCL on GPUs, gloo on CPU).  The all-to-all takes split sizes on the
host, so each forward reads the M x N keep matrix back once (a sync-free variant would
write rows straight into capacity-shaped receive buffers on the peers).
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Callable, List, Optional

import torch

from . import _native as nat


@dataclasses.dataclass
class EpPlan:
    rank: int
    world: int
    rho: List[int]
    keep: torch.Tensor       # [M, N] int32: kept routes of split (source s, expert e)
    recv_off: torch.Tensor   # [M, N] int32: first row of split (s, e) in rho(e)'s buffer
    R_req: torch.Tensor      # [M] requested rows per destination (Eq. 20)
    R_keep: torch.Tensor     # [M] kept rows per destination (Eq. 21)
    dst_row: torch.Tensor    # [T, K] int32: row of the route in rho(e)'s buffer, -1 dropped
    send_pos: torch.Tensor   # [T, K] int32: row of the route in this rank's send buffer, -1
    keep_host: torch.Tensor  # [M, N] int64 copy of keep on the host (the split sizes)

    def local_offsets(self) -> torch.Tensor:
        """Eq. 26 over this rank's experts in ascending index: [n_local + 1] int32 (host)."""
        sizes = [int(self.keep_host[:, e].sum()) for e in range(self.keep_host.shape[1])
                 if self.rho[e] == self.rank]
        off = [0]
        for m in sizes:
            off.append(off[-1] + m)
        return torch.tensor(off, dtype=torch.int32)

    def send_counts(self) -> torch.Tensor:
        """[M, M] host: rows source s sends to destination q (from the keep matrix alone)."""
        out = torch.zeros((self.world, self.world), dtype=torch.int64)
        for e, q in enumerate(self.rho):
            out[:, q] += self.keep_host[:, e]
        return out


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _rho(rho):
    return (ctypes.c_int32 * len(rho))(*[int(v) for v in rho])


def gather_counts(counts_local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of the N-length requested split counts: [M, N] (the device of the input)."""
    import torch.distributed as dist
    M = dist.get_world_size(group)
    parts = [torch.empty_like(counts_local) for _ in range(M)]
    dist.all_gather(parts, counts_local.contiguous(), group=group)
    return torch.stack(parts).to(torch.int32).contiguous()


def make_plan(counts_all: torch.Tensor, topk_idx: torch.Tensor, rank: int, K: int, rho: List[int],
              cap_policy: str = "rank_wide", capacity_factor: float = 1.0,
              route_pos: Optional[torch.Tensor] = None, offsets: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, stream=None) -> EpPlan:
    """The keep matrix, this rank's destination rows and send positions.  CUDA tensors use the
    device entries (route_pos / offsets of a capacity-free moe_permute of the rank's batch and
    a layer workspace are then required); CPU tensors use the host entries."""
    lib = nat.library()
    M, N = counts_all.shape
    T = topk_idx.shape[0]
    pol = nat.CAP_POLICIES[cap_policy] if isinstance(cap_policy, str) else int(cap_policy)
    rho_arr = _rho(rho)
    dev = counts_all.device
    keep = torch.empty((M, N), dtype=torch.int32, device=dev)
    recv_off = torch.empty((M, N), dtype=torch.int32, device=dev)
    R_req = torch.empty((M,), dtype=torch.int32, device=dev)
    R_keep = torch.empty((M,), dtype=torch.int32, device=dev)
    dst_row = torch.empty((T, K), dtype=torch.int32, device=dev)
    send_pos = torch.empty((T, K), dtype=torch.int32, device=dev)
    if dev.type == "cuda":
        st = nat._stream(stream)
        nat._check("moe_ep_keep_matrix", lib.moe_ep_keep_matrix(
            M, N, K, rho_arr, pol, float(capacity_factor), _ptr(counts_all), _ptr(keep),
            _ptr(recv_off), _ptr(R_req), _ptr(R_keep), st))
        nat._check("moe_ep_place", lib.moe_ep_place(
            M, rank, T, N, K, _ptr(topk_idx), _ptr(route_pos), _ptr(offsets), _ptr(keep),
            _ptr(recv_off), _ptr(dst_row), _ptr(workspace), workspace.numel(), st))
        nat._check("moe_ep_send_pos", lib.moe_ep_send_pos(
            M, rank, T, N, K, rho_arr, _ptr(topk_idx), _ptr(keep), _ptr(recv_off), _ptr(dst_row),
            _ptr(send_pos), None, _ptr(workspace), workspace.numel(), st))
    else:
        counts_all = counts_all.to(torch.int32).contiguous()
        nat._check("moe_ep_keep_matrix_host", lib.moe_ep_keep_matrix_host(
            M, N, K, rho_arr, pol, float(capacity_factor), _ptr(counts_all), _ptr(keep),
            _ptr(recv_off), _ptr(R_req), _ptr(R_keep)))
        idx = topk_idx.to(torch.int32).contiguous()
        nat._check("moe_ep_place_host", lib.moe_ep_place_host(
            M, rank, T, N, K, _ptr(idx), _ptr(keep), _ptr(recv_off), _ptr(dst_row)))
        nat._check("moe_ep_send_pos_host", lib.moe_ep_send_pos_host(
            M, rank, T, N, K, rho_arr, _ptr(idx), _ptr(keep), _ptr(recv_off), _ptr(dst_row),
            _ptr(send_pos), None))
    return EpPlan(rank, M, list(rho), keep, recv_off, R_req, R_keep, dst_row, send_pos,
                  keep.cpu().to(torch.int64))


def rows_copy(src: torch.Tensor, dst: torch.Tensor, n: int, src_index=None, src_div: int = 1,
              dst_index=None, zero_missing: bool = False, workspace=None, stream=None):
    """dst[dst_index[i]] = src[src_index[i]] for i < n (moe_rows_copy; see the C header):
    row-major 2-D tensors of the same row width, device or host alike."""
    lib = nat.library()
    row_bytes = src.shape[1] * src.element_size()
    if src.device.type == "cuda":
        nat._check("moe_rows_copy", lib.moe_rows_copy(
            _ptr(src), src.shape[0], _ptr(src_index), src_div, _ptr(dst), dst.shape[0],
            _ptr(dst_index), n, row_bytes, 1 if zero_missing else 0, _ptr(workspace),
            workspace.numel(), nat._stream(stream)))
    else:
        nat._check("moe_rows_copy_host", lib.moe_rows_copy_host(
            _ptr(src), src.shape[0], _ptr(src_index), src_div, _ptr(dst), dst.shape[0],
            _ptr(dst_index), n, row_bytes, 1 if zero_missing else 0))


def recv_rows(plan: EpPlan, workspace=None, stream=None) -> torch.Tensor:
    """Row of this rank's packed buffer for each row of its receive buffer (moe_ep_recv_rows)."""
    lib = nat.library()
    M, N = plan.keep.shape
    n = int(plan.send_counts()[:, plan.rank].sum())
    out = torch.empty((n,), dtype=torch.int32, device=plan.keep.device)
    if plan.keep.device.type == "cuda":
        nat._check("moe_ep_recv_rows", lib.moe_ep_recv_rows(
            M, plan.rank, N, _rho(plan.rho), _ptr(plan.keep), _ptr(plan.recv_off), _ptr(out), n,
            _ptr(workspace), workspace.numel(), nat._stream(stream)))
    else:
        nat._check("moe_ep_recv_rows_host", lib.moe_ep_recv_rows_host(
            M, plan.rank, N, _rho(plan.rho), _ptr(plan.keep), _ptr(plan.recv_off), _ptr(out), n))
    return out


@dataclasses.dataclass
class Dispatched:
    rows: torch.Tensor            # [R_keep[rank], d] this rank's packed buffer
    recv_row: torch.Tensor        # [n_recv] packed row of each received row
    send_split: List[int]         # rows sent to each destination
    recv_split: List[int]         # rows received from each source


def dispatch(x_local: torch.Tensor, plan: EpPlan, K: int, group=None, workspace=None,
             stream=None) -> Dispatched:
    """Send every kept route's token row to its row of rank rho(e)'s packed buffer."""
    import torch.distributed as dist
    counts = plan.send_counts()
    me = plan.rank
    send_split = [int(v) for v in counts[me].tolist()]
    recv_split = [int(v) for v in counts[:, me].tolist()]
    T, d = x_local.shape
    send = torch.empty((sum(send_split), d), dtype=x_local.dtype, device=x_local.device)
    rows_copy(x_local, send, T * K, src_div=K, dst_index=plan.send_pos, workspace=workspace,
              stream=stream)
    recv = torch.empty((sum(recv_split), d), dtype=x_local.dtype, device=x_local.device)
    dist.all_to_all_single(recv, send, recv_split, send_split, group=group)
    rr = recv_rows(plan, workspace, stream)
    rows = torch.empty((int(plan.keep_host[:, [e for e in range(len(plan.rho))
                                                if plan.rho[e] == me]].sum()), d),
                       dtype=x_local.dtype, device=x_local.device)
    rows_copy(recv, rows, recv.shape[0], dst_index=rr, workspace=workspace, stream=stream)
    return Dispatched(rows, rr, send_split, recv_split)


def return_outputs(f_packed: torch.Tensor, plan: EpPlan, disp: Dispatched, T: int, K: int,
                   group=None, workspace=None, stream=None) -> torch.Tensor:
    """The reverse exchange: the output row of every received route goes back to its source.
    Returns [T * K, d] on each source: row t * K + k is route (t, k)'s expert output, zero for
    dropped routes."""
    import torch.distributed as dist
    d = f_packed.shape[1]
    send = torch.empty((disp.recv_row.shape[0], d), dtype=f_packed.dtype, device=f_packed.device)
    rows_copy(f_packed, send, send.shape[0], src_index=disp.recv_row, workspace=workspace,
              stream=stream)
    back = torch.empty((sum(disp.send_split), d), dtype=f_packed.dtype, device=f_packed.device)
    dist.all_to_all_single(back, send, disp.send_split, disp.recv_split, group=group)
    out = torch.empty((T * K, d), dtype=f_packed.dtype, device=f_packed.device)
    rows_copy(back, out, T * K, src_index=plan.send_pos, zero_missing=True, workspace=workspace,
              stream=stream)
    return out


def ep_layer_forward(x_local: torch.Tensor, topk_idx: torch.Tensor, rho: List[int], K: int,
                     expert_fn: Callable[[torch.Tensor, torch.Tensor], torch.Tensor],
                     merge_fn: Callable[[torch.Tensor, torch.Tensor], torch.Tensor],
                     counts_local: torch.Tensor, cap_policy: str = "rank_wide",
                     capacity_factor: float = 1.0, group=None, **plan_kw):
    """Steps 2-5 for this rank's tokens, given its routing (topk_idx [T, K] and the count
    vector of its requests).  expert_fn(rows, local_offsets) computes the outputs of this
    rank's packed buffer (local experts in ascending index, segments local_offsets; rows
    holds exactly R_keep[rank] rows, so a grouped GEMM whose configuration expects a buffer
    of T' K rows gets them copied into one of that size);
    merge_fn(route_out [T*K, d], kept [T, K]) merges them into y (Eq. 80).
    Returns (y, plan)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    counts_all = gather_counts(counts_local, group)
    plan = make_plan(counts_all, topk_idx, rank, K, rho, cap_policy, capacity_factor, **plan_kw)
    ws, st = plan_kw.get("workspace"), plan_kw.get("stream")
    disp = dispatch(x_local, plan, K, group, ws, st)
    f_packed = expert_fn(disp.rows, plan.local_offsets())
    route_out = return_outputs(f_packed, plan, disp, x_local.shape[0], K, group, ws, st)
    return merge_fn(route_out, plan.dst_row >= 0), plan
