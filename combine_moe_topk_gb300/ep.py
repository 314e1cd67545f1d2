"""Expert-parallel exchange of the MoE token path: R ranks, one GPU each,
rank r owning experts [r*E, (r+1)*E), E = e / R.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all", description: a token goes to each destination rank once, not
once per selected expert (about 1.29x of its gain on its own); the transport
takes tokens before the top-k expansion and replicates them itself, groups
the arrivals by expert for the grouped GEMM, and reduces in its combine; the
gradient of a combine is a dispatch and the gradient of a dispatch is a
combine, against the forward's handle.  Review thread: the routing weights
travel with the tokens and are applied on the expert's rank (the combine
sums rows, it does not weight them); the row counts come from the host, not
from a device read in front of every GEMM; every rank must agree on sizes.

One layer, forward (all device work in the library's kernels):

    source  h = moe_dispatch_layout_ex(idx, e, R virtual ranks, send_slots)
            plan = exchange_counts(h)          one all-to-all of R counts and
                                               the only host read of the layout;
                                               backward and replays reuse it
            send = source_send(h, x, gate, plan)     moe_ep_pack + moe_ep_dispatch
    all-to-all: the rows, their local expert ids and gates
    dest    recv = dest_receive(rows, ids, gates, E) layout of the arrivals
                                               (absent routes), moe_dispatch
            expert(recv.X) -> y                grouped rows, e.g. moe_grouped_gemm
            P = dest_partial(recv, y)          moe_combine with the gates
    all-to-all back: P
    source  out = source_reduce(h, send, P)    moe_ep_combine (rank-order sum)

and backward: dout goes out like x (source_send_grad), the destination runs
moe_combine_bwd (dY for the expert's backward, the gate gradients sent back,
source_dgate), the expert's input gradient is summed per arrival
(dest_dispatch_bwd) and comes back like P (source_reduce).

The transport is ``torch.distributed.all_to_all_single`` on the given group
(NCCL between GPUs; any backend that has all-to-all works, so the plan and
the exchange run on CPU tensors over gloo as well).  Every phase function is
one rank's side; ExpertParallelMoE strings them together for a process
group.  A batch of s tokens per rank sends at most s*R rows.
"""
from __future__ import annotations

import dataclasses

import torch

from . import binding as B


@dataclasses.dataclass
class Plan:
    """Sizes of one layout's exchange on this rank (host integers)."""
    send_counts: list   # rows (tokens) to each destination rank, in rank order
    recv_counts: list   # rows (tokens) from each source rank, in rank order
    recv_routes: list | None = None  # kept routes from each source to this rank's experts

    @property
    def rows_sent(self) -> int:
        return sum(self.send_counts)

    @property
    def rows_recv(self) -> int:
        return sum(self.recv_counts)

    @property
    def routes_recv(self) -> int:
        """Rows of this rank's grouped buffer (0 when not exchanged)."""
        return sum(self.recv_routes) if self.recv_routes is not None else 0


def route_counts(h: B.Handle) -> torch.Tensor:
    """Kept routes to each virtual rank's experts ([R], from the handle's counts)."""
    return h.counts().view(h.R, h.e // h.R).sum(dim=1)


def exchange_counts(rank_counts: torch.Tensor, group=None, routes: torch.Tensor | None = None) -> Plan:
    """All-to-all of this rank's per-destination token counts ([R] int32,
    e.g. a layout handle's rank_counts) -- and, given, its kept routes to
    each destination -- into a Plan.  Reads the counts on the host once
    (the exchange and the receiving buffers are sized by them)."""
    import torch.distributed as dist

    cols = [rank_counts.to(torch.int64)] + ([routes.to(torch.int64)] if routes is not None else [])
    send = torch.stack(cols, dim=1).contiguous()  # [R, 1 or 2]: row r goes to rank r
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    s, r = send.tolist(), recv.tolist()
    return Plan(send_counts=[int(v[0]) for v in s], recv_counts=[int(v[0]) for v in r],
                recv_routes=[int(v[1]) for v in r] if routes is not None else None)


def all_to_all(t: torch.Tensor, plan: Plan, group=None, back: bool = False) -> torch.Tensor:
    """Rows of t go to the ranks the plan says: forward sends send_counts
    rows to each rank and receives recv_counts rows from each; back is the
    reverse exchange (the partials and gradients returning to their source)."""
    import torch.distributed as dist

    out_counts, in_counts = (plan.send_counts, plan.recv_counts) if back else (plan.recv_counts, plan.send_counts)
    out = torch.empty((sum(out_counts),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    dist.all_to_all_single(out, t.contiguous(), out_counts, in_counts, group=group)
    return out


@dataclasses.dataclass
class Send:
    """A source rank's side of one layout's exchange."""
    send_row: torch.Tensor   # [s, R] int32: row of each token in each destination segment, -1 = not sent
    rows_sent: int
    X_send: torch.Tensor | None = None
    meta_idx: torch.Tensor | None = None   # [rows_sent, k] local expert ids as the destination sees them
    meta_gate: torch.Tensor | None = None  # [rows_sent, k] their gates


def source_send(h: B.Handle, x: torch.Tensor, gate: torch.Tensor, plan: Plan) -> Send:
    """The send buffer and its routing metadata: each token row once per
    destination rank that holds one of its kept routes."""
    if h.R != len(plan.send_counts):
        raise B.MoEError(1, "source_send", f"handle has {h.R} virtual ranks, plan {len(plan.send_counts)}")
    send_row, meta_idx, meta_gate = B.moe_ep_pack(h, gate, plan.rows_sent)
    X_send = B.moe_ep_dispatch(h, send_row, plan.rows_sent, x)
    return Send(send_row=send_row, rows_sent=plan.rows_sent, X_send=X_send, meta_idx=meta_idx, meta_gate=meta_gate)


@dataclasses.dataclass
class Recv:
    """A destination rank's arrivals, grouped by its local experts."""
    h: B.Handle               # layout of the arrivals over the E local experts (absent routes allowed)
    X: torch.Tensor           # [h.rows, m] grouped rows (expert segments at h.offsets())
    meta_gate: torch.Tensor   # [arrivals, k] the routes' gates


def dest_receive(rows: torch.Tensor, meta_idx: torch.Tensor, meta_gate: torch.Tensor, E: int,
                 routes: int = 0) -> Recv:
    """Group the arrivals (from source 0, 1, ... in order) by local expert;
    routes (the plan's routes_recv) sizes the grouped buffer exactly, else it
    is the bound arrivals * k."""
    hr = B.moe_dispatch_layout_ex(meta_idx, E, absent_routes=True, rows_bound=routes)
    return Recv(h=hr, X=B.moe_dispatch(hr, rows), meta_gate=meta_gate)


def dest_partial(recv: Recv, y: torch.Tensor) -> torch.Tensor:
    """Each arrival's weighted sum over its routes to this rank's experts."""
    return B.moe_combine(recv.h, y, recv.meta_gate)


def source_reduce(h: B.Handle, send: Send, P_back: torch.Tensor) -> torch.Tensor:
    """The returned rows summed per token over destination ranks, in rank order."""
    return B.moe_ep_combine(h, send.send_row, send.rows_sent, P_back)


def source_send_grad(h: B.Handle, send: Send, dout: torch.Tensor) -> torch.Tensor:
    """The combine's gradient goes out like the tokens did."""
    return B.moe_ep_dispatch(h, send.send_row, send.rows_sent, dout)


def dest_combine_bwd(recv: Recv, dP: torch.Tensor, y: torch.Tensor):
    """(dY [rows, m] for the expert's backward, the arrivals' gate gradients [arrivals, k])."""
    return B.moe_combine_bwd(recv.h, dP, recv.meta_gate, y)


def dest_dispatch_bwd(recv: Recv, dX: torch.Tensor) -> torch.Tensor:
    """Each arrival's input gradient: its grouped rows' gradients summed."""
    return B.moe_dispatch_bwd(recv.h, dX)


def source_dgate(h: B.Handle, send: Send, dgate_back: torch.Tensor) -> torch.Tensor:
    """The source's gate gradients from the ones its destinations returned."""
    return B.moe_ep_unpack_dgate(h, send.send_row, send.rows_sent, dgate_back)


class ExpertParallelMoE:
    """One rank's expert-parallel MoE layer over a process group of R ranks:
    forward and backward of dispatch -> expert -> weighted combine, with the
    expert given as a pair of functions on the grouped rows (its forward,
    and its backward from dY to dX).  ``layout`` builds the source handle
    once per batch; ``forward`` / ``backward`` replay it (the plan's counts
    are read on the host once per layout, at ``layout``)."""

    def __init__(self, e: int, group=None):
        import torch.distributed as dist

        self.group = group
        self.R = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if e % self.R:
            raise ValueError(f"{e} experts do not split over {self.R} ranks")
        self.e, self.E = e, e // self.R

    def layout(self, idx: torch.Tensor, capacity: int = 0) -> tuple[B.Handle, Plan]:
        h = B.moe_dispatch_layout_ex(idx, self.e, capacity, self.R, send_slots=True)
        return h, exchange_counts(h.rank_counts(), self.group, route_counts(h))

    def forward(self, h: B.Handle, plan: Plan, x: torch.Tensor, gate: torch.Tensor, expert_fwd):
        send = source_send(h, x, gate, plan)
        rows = all_to_all(send.X_send, plan, self.group)
        ids = all_to_all(send.meta_idx, plan, self.group)
        gates = all_to_all(send.meta_gate, plan, self.group)
        recv = dest_receive(rows, ids, gates, self.E, plan.routes_recv)
        y = expert_fwd(recv)
        P = dest_partial(recv, y)
        out = source_reduce(h, send, all_to_all(P, plan, self.group, back=True))
        return out, (send, recv, y)

    def backward(self, h: B.Handle, plan: Plan, saved, dout: torch.Tensor, expert_bwd):
        send, recv, y = saved
        dP = all_to_all(source_send_grad(h, send, dout), plan, self.group)
        dY, dg_recv = dest_combine_bwd(recv, dP, y)
        dgate = source_dgate(h, send, all_to_all(dg_recv, plan, self.group, back=True))
        dX = expert_bwd(recv, dY)
        dx = source_reduce(h, send, all_to_all(dest_dispatch_bwd(recv, dX), plan, self.group, back=True))
        return dx, dgate
