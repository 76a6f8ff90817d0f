"""Expert parallelism across ranks: capacity agreement, dispatch and combine.

Section 10 "Routing, Capacity, and Load Balancing", Section 10.3 (Eq. 23 and Eq. 26,
Figure 41).  Each rank holds a batch of tokens and the experts rho maps to it.  Per forward:

1. each rank routes its own tokens and counts its requests per expert (C^req of its batch);
2. the ranks all-gather those N-length count vectors; each derives the same keep matrix and
   the destination row of each of its routes (``moe_ep_keep_matrix`` / ``moe_ep_place`` on
   CUDA tensors, their host twins on CPU tensors): destination q packs, per local expert in
   ascending index, the kept rows of source 0, then source 1, ...;
3. dispatch: every kept route's token row goes to rank rho(e), row dst_row of its buffer
   (one all-to-all of rows and their destination rows, then a scatter);
4. each rank runs its local experts over its packed buffer (segments from the keep matrix);
5. combine: the expert outputs go back to their sources (the reverse all-to-all), and each
   source merges them with its shared branch (Eq. 80; dropped routes add nothing).

This module plans and moves data; the routing, the expert GEMMs and the merge are callables
(on a GPU: the library's kernels).  The collectives are ``torch.distributed`` (NCCL on GPUs,
gloo on CPU).  The all-to-all takes split sizes on the host, so each forward reads the M x M
send counts back once (a sync-free variant would write rows straight into capacity-shaped
receive buffers on the peers).
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

    def local_offsets(self) -> torch.Tensor:
        """Eq. 26 over this rank's experts in ascending index: [n_local + 1] int32 (host)."""
        keep = self.keep.cpu()
        sizes = [int(keep[:, e].sum()) for e in range(keep.shape[1]) if self.rho[e] == self.rank]
        off = [0]
        for m in sizes:
            off.append(off[-1] + m)
        return torch.tensor(off, dtype=torch.int32)

    def send_counts(self) -> torch.Tensor:
        """[M, M] host: rows source s sends to destination q (from the keep matrix alone)."""
        keep = self.keep.cpu().to(torch.int64)
        M = self.world
        out = torch.zeros((M, M), dtype=torch.int64)
        for e, q in enumerate(self.rho):
            out[:, q] += keep[:, e]
        return out


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


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
    """The keep matrix and this rank's destination rows.  CUDA tensors use the device
    entries (route_pos / offsets of a capacity-free moe_permute of the rank's batch and a
    layer workspace are then required); CPU tensors use the host entries."""
    lib = nat.library()
    M, N = counts_all.shape
    T = topk_idx.shape[0]
    pol = nat.CAP_POLICIES[cap_policy] if isinstance(cap_policy, str) else int(cap_policy)
    rho_arr = (ctypes.c_int32 * N)(*[int(v) for v in rho])
    dev = counts_all.device
    keep = torch.empty((M, N), dtype=torch.int32, device=dev)
    recv_off = torch.empty((M, N), dtype=torch.int32, device=dev)
    R_req = torch.empty((M,), dtype=torch.int32, device=dev)
    R_keep = torch.empty((M,), dtype=torch.int32, device=dev)
    dst_row = torch.empty((T, K), dtype=torch.int32, device=dev)
    if dev.type == "cuda":
        nat._check("moe_ep_keep_matrix", lib.moe_ep_keep_matrix(
            M, N, K, rho_arr, pol, float(capacity_factor), _ptr(counts_all), _ptr(keep),
            _ptr(recv_off), _ptr(R_req), _ptr(R_keep), nat._stream(stream)))
        nat._check("moe_ep_place", lib.moe_ep_place(
            M, rank, T, N, K, _ptr(topk_idx), _ptr(route_pos), _ptr(offsets), _ptr(keep),
            _ptr(recv_off), _ptr(dst_row), _ptr(workspace), workspace.numel(), nat._stream(stream)))
    else:
        counts_all = counts_all.to(torch.int32).contiguous()
        nat._check("moe_ep_keep_matrix_host", lib.moe_ep_keep_matrix_host(
            M, N, K, rho_arr, pol, float(capacity_factor), _ptr(counts_all), _ptr(keep),
            _ptr(recv_off), _ptr(R_req), _ptr(R_keep)))
        idx = topk_idx.to(torch.int32).contiguous()
        nat._check("moe_ep_place_host", lib.moe_ep_place_host(
            M, rank, T, N, K, _ptr(idx), _ptr(keep), _ptr(recv_off), _ptr(dst_row)))
    return EpPlan(rank, M, list(rho), keep, recv_off, R_req, R_keep, dst_row)


@dataclasses.dataclass
class Dispatched:
    rows: torch.Tensor            # [R_keep[rank], d] this rank's packed buffer
    sent_routes: torch.Tensor     # [n_sent] flat route index (t * K + k) of each sent row
    send_split: List[int]         # rows sent to each destination
    recv_split: List[int]         # rows received from each source
    recv_rows: torch.Tensor       # [n_recv] packed row of each received row


def dispatch(x_local: torch.Tensor, plan: EpPlan, topk_idx: torch.Tensor, group=None) -> Dispatched:
    """Send every kept route's token row to row dst_row of rank rho(e)'s packed buffer."""
    import torch.distributed as dist
    M, me = plan.world, plan.rank
    K = topk_idx.shape[1]
    rho_t = torch.tensor(plan.rho, dtype=torch.int64, device=x_local.device)
    flat_e = topk_idx.reshape(-1).to(torch.int64)
    flat_row = plan.dst_row.reshape(-1).to(torch.int64)
    kept = flat_row >= 0
    dest = torch.where(kept, rho_t[flat_e.clamp(min=0)], torch.full_like(flat_e, M))
    # kept routes grouped by destination, each group in destination-row order
    order = torch.argsort(dest * (1 << 40) + flat_row.clamp(min=0), stable=True)
    order = order[: int(kept.sum())]
    counts = plan.send_counts()
    send_split = [int(v) for v in counts[me].tolist()]
    recv_split = [int(v) for v in counts[:, me].tolist()]
    send_rows = x_local[order // K].contiguous()
    send_idx = flat_row[order].contiguous()
    d = x_local.shape[1]
    recv = torch.empty((sum(recv_split), d), dtype=x_local.dtype, device=x_local.device)
    recv_idx = torch.empty((sum(recv_split),), dtype=torch.int64, device=x_local.device)
    dist.all_to_all_single(recv, send_rows, recv_split, send_split, group=group)
    dist.all_to_all_single(recv_idx, send_idx, recv_split, send_split, group=group)
    n_local = int(plan.R_keep.cpu()[me])
    rows = torch.empty((n_local, d), dtype=x_local.dtype, device=x_local.device)
    rows[recv_idx] = recv
    return Dispatched(rows, order, send_split, recv_split, recv_idx)


def return_outputs(f_packed: torch.Tensor, disp: Dispatched, T: int, K: int, group=None) -> torch.Tensor:
    """The reverse exchange: the output row of every received route goes back to its
    source.  Returns [T * K, d] on each source: row t * K + k is route (t, k)'s expert
    output, zero for dropped routes."""
    import torch.distributed as dist
    send = f_packed[disp.recv_rows].contiguous()
    back = torch.empty((sum(disp.send_split), f_packed.shape[1]), dtype=f_packed.dtype,
                       device=f_packed.device)
    dist.all_to_all_single(back, send, disp.send_split, disp.recv_split, group=group)
    out = torch.zeros((T * K, f_packed.shape[1]), dtype=f_packed.dtype, device=f_packed.device)
    out[disp.sent_routes] = back
    return out


def ep_layer_forward(x_local: torch.Tensor, topk_idx: torch.Tensor, rho: List[int], K: int,
                     expert_fn: Callable[[torch.Tensor, torch.Tensor], torch.Tensor],
                     merge_fn: Callable[[torch.Tensor, torch.Tensor], torch.Tensor],
                     counts_local: torch.Tensor, cap_policy: str = "rank_wide",
                     capacity_factor: float = 1.0, group=None, **plan_kw):
    """Steps 2-5 for this rank's tokens, given its routing (topk_idx [T, K] and the count
    vector of its requests).  expert_fn(rows, local_offsets) computes the outputs of this
    rank's packed buffer (local experts in ascending index, segments local_offsets);
    merge_fn(route_out [T*K, d], kept [T, K]) merges them into y (Eq. 80).
    Returns (y, plan)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    counts_all = gather_counts(counts_local, group)
    plan = make_plan(counts_all, topk_idx, rank, K, rho, cap_policy, capacity_factor, **plan_kw)
    disp = dispatch(x_local, plan, topk_idx, group)
    f_packed = expert_fn(disp.rows, plan.local_offsets())
    route_out = return_outputs(f_packed, disp, x_local.shape[0], K, group)
    return merge_fn(route_out, plan.dst_row >= 0), plan
