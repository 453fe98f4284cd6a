"""Expert-parallel MoE layer across ranks: dispatch of routed rows to the
ranks that hold their experts, and the return exchange before the top-k
combine (matmul_ogs.py: FusedComm, post_matmul_comm_torch).

Rank r of G holds experts [r*E_loc, (r+1)*E_loc).  Every step on the data
runs in libgg.so's kernels (route, permute, the receive-side row map, the
combine); the exchanges are the caller's collectives, by default
``torch.distributed.all_to_all_single`` (NCCL for CUDA tensors, gloo for CPU
tensors).  The one host synchronisation is the read of the count matrices
that the variable-size row exchange needs as split sizes.

Each exchange-free step is a method of its own (``dispatch_local``,
``dispatch_plan``, ``dispatch_finish``, ``combine_local``,
``combine_finish``), so a caller with its own transport can interleave them
with its exchanges; ``dispatch`` and ``combine`` chain them through
``self.exchange``.
"""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np
import torch

from . import _lib, api


class TorchDistExchange:
    """Exchanges through torch.distributed (the default process group unless one is given)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def all_to_all_equal(self, out, inp):
        self.dist.all_to_all_single(out, inp, group=self.group)

    def all_to_all(self, out, inp, out_splits, in_splits):
        self.dist.all_to_all_single(out, inp, [int(c) for c in out_splits], [int(c) for c in in_splits],
                                    group=self.group)


def plan(m_sizes, recv_m, G: int, E_loc: int, row_map: bool = False) -> dict:
    """Host plan through gg_ep_plan: m_sizes [G*E_loc] (this rank's histogram),
    recv_m [G, E_loc] (counts received from every rank).  Returns send_counts
    [G], recv_counts [G] (int64), local_m_sizes [E_loc] (int32) and, on
    request, row_map [R_loc] (int32), all numpy."""
    m = np.ascontiguousarray(np.asarray(m_sizes, dtype=np.int32).reshape(-1))
    rm = np.ascontiguousarray(np.asarray(recv_m, dtype=np.int32).reshape(-1))
    if m.size != G * E_loc or rm.size != G * E_loc:
        raise ValueError("m_sizes and recv_m must have G*E_loc entries")
    send = np.zeros(G, np.int64)
    recv = np.zeros(G, np.int64)
    loc = np.zeros(E_loc, np.int32)
    R_loc = int(rm.astype(np.int64).sum())
    rmap = np.zeros(R_loc, np.int32) if row_map else None
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = _lib.load().gg_ep_plan(p(m), p(rm), G, E_loc, p(send), p(recv), p(loc), p(rmap),
                                R_loc if row_map else 0)
    _lib.check("gg_ep_plan", rc)
    return dict(send_counts=send, recv_counts=recv, local_m_sizes=loc, row_map=rmap)


def recv_map(recv_m_dev, G: int, E_loc: int, R_loc: int, *, out=None, status=None):
    """row_map [R_loc] int32 on the device from the device count matrix [G, E_loc]."""
    api._need(recv_m_dev, torch.int32, "recv_m", (G, E_loc))
    rmap = api._out(out, (R_loc,), torch.int32, recv_m_dev.device, "out")
    rc = _lib.load().gg_ep_recv_map(api._p(recv_m_dev), G, E_loc, R_loc, api._p(rmap), api._p(status),
                                    api._stream(recv_m_dev.device))
    _lib.check("gg_ep_recv_map", rc)
    return rmap


@dataclasses.dataclass
class Dispatched:
    """One rank's view of a dispatched batch."""
    x: torch.Tensor            # [R_loc, K] rows for this rank's experts, expert-contiguous
    m_sizes: torch.Tensor      # [E_loc] int32 (device), rows per local expert
    row_map: torch.Tensor      # [R_loc] int32: received row -> local expert-order row
    route: dict                # this rank's own routing (m_sizes over all E, gather_idx, row_id_map)
    send_counts: list          # rows sent to each rank
    recv_counts: list          # rows received from each rank
    T: int
    topk: int
    y_back: torch.Tensor | None = None  # the combine's input, kept for its backward


class ExpertParallel:
    """Expert-parallel dispatch/combine for rank `rank` of `world_size`, E experts in all."""

    def __init__(self, E: int, rank: int, world_size: int, exchange=None):
        if E % world_size:
            raise ValueError("E must be a multiple of the number of ranks")
        self.E, self.rank, self.G = E, rank, world_size
        self.E_loc = E // world_size
        self.exchange = exchange if exchange is not None else TorchDistExchange()

    # ---------------------------------------------------------- dispatch --
    def dispatch_local(self, X, topk_ids, status=None):
        """Route this rank's tokens over all E experts and permute them into
        expert order.  Returns (route, Xp, counts [G, E_loc] device int32)."""
        T, topk = topk_ids.shape
        r = api.route_hist_offsets(topk_ids, self.E, status=status)
        Xp = api.permute(X, r["row_id_map"], topk, status=status)
        return r, Xp, r["m_sizes"].view(self.G, self.E_loc)

    def dispatch_plan(self, counts, recv_m):
        """Host plan from this rank's counts and the received count matrix."""
        return plan(counts.cpu().numpy(), recv_m.cpu().numpy(), self.G, self.E_loc)

    def dispatch_finish(self, x_recv, recv_m, pl, route, T, topk, status=None) -> Dispatched:
        """Received rows (source after source) into local expert order."""
        R_loc = x_recv.shape[0]
        rmap = recv_map(recv_m, self.G, self.E_loc, R_loc, status=status)
        x_loc = api.permute(x_recv, rmap, 1, status=status)
        m_loc = torch.from_numpy(pl["local_m_sizes"]).to(x_recv.device)
        return Dispatched(x=x_loc, m_sizes=m_loc, row_map=rmap, route=route,
                          send_counts=[int(c) for c in pl["send_counts"]],
                          recv_counts=[int(c) for c in pl["recv_counts"]], T=T, topk=topk)

    def dispatch(self, X, topk_ids, status=None) -> Dispatched:
        T, topk = topk_ids.shape
        route, Xp, counts = self.dispatch_local(X, topk_ids, status)
        recv_m = torch.empty_like(counts)
        self.exchange.all_to_all_equal(recv_m, counts)
        pl = self.dispatch_plan(counts, recv_m)
        x_recv = torch.empty(int(pl["recv_counts"].sum()), X.shape[1], dtype=X.dtype, device=X.device)
        self.exchange.all_to_all(x_recv, Xp, pl["recv_counts"], pl["send_counts"])
        return self.dispatch_finish(x_recv, recv_m, pl, route, T, topk, status)

    # ----------------------------------------------------------- combine --
    def combine_local(self, y_loc, d: Dispatched, status=None):
        """Local expert-order results back into received order."""
        return api.unpermute_combine(y_loc, d.row_map, None, y_loc.shape[0], 1, status=status)

    def combine_finish(self, y_back, d: Dispatched, topk_w=None, status=None):
        """Returned rows (this rank's expert order) -> weighted top-k combine."""
        d.y_back = y_back
        return api.unpermute_combine(y_back, d.route["row_id_map"], topk_w, d.T, d.topk, status=status)

    def combine(self, y_loc, d: Dispatched, topk_w=None, status=None):
        """out [T, N]: the local experts' results, sent back and combined."""
        y_recv = self.combine_local(y_loc, d, status)
        y_back = torch.empty(sum(d.send_counts), y_loc.shape[1], dtype=y_loc.dtype, device=y_loc.device)
        self.exchange.all_to_all(y_back, y_recv, d.send_counts, d.recv_counts)
        return self.combine_finish(y_back, d, topk_w, status)

    # ---------------------------------------------------------- backward --
    def combine_backward(self, grad_out, d: Dispatched, topk_w=None, status=None):
        """(dy_loc [R_loc, N], dw [T, topk] or None): the gradient of combine
        with respect to the local results and the routing weights (dw needs the
        forward's combine input, kept by combine)."""
        dy_back, dw = api.unpermute_combine_bwd(grad_out, d.y_back, d.route["row_id_map"], topk_w, d.T,
                                                d.topk, want_dw=d.y_back is not None, status=status)
        dy_recv = torch.empty(sum(d.recv_counts), dy_back.shape[1], dtype=dy_back.dtype,
                              device=dy_back.device)
        self.exchange.all_to_all(dy_recv, dy_back, d.recv_counts, d.send_counts)
        return api.permute(dy_recv, d.row_map, 1, status=status), dw

    def dispatch_backward(self, dx_loc, d: Dispatched, status=None):
        """dX [T, K]: the gradient of dispatch, each token's slots summed."""
        dx_recv = api.unpermute_combine(dx_loc, d.row_map, None, dx_loc.shape[0], 1, status=status)
        dx_back = torch.empty(sum(d.send_counts), dx_loc.shape[1], dtype=dx_loc.dtype, device=dx_loc.device)
        self.exchange.all_to_all(dx_back, dx_recv, d.send_counts, d.recv_counts)
        return api.unpermute_combine(dx_back, d.route["row_id_map"], None, d.T, d.topk, status=status)
