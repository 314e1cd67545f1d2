"""Expert-parallel exchange of the token path over R ranks, as plain CPU
code: the oracle of the library's expert-parallel steps.

TEST INFRASTRUCTURE ONLY: the test-suite and the benchmark's CPU legs are its
only callers; the product package never imports it.  It is built from the
C oracle's pinned primitives (layout, send slots, dispatch, combine and
their backwards) and NumPy permutations for the exchange, in the order the
method takes the steps.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all", description: a token goes to each destination rank once, not
once per selected expert; the transport takes tokens before the top-k
expansion and replicates them itself, groups the arrivals by expert for the
grouped GEMM, and reduces in its combine; the gradient of a combine is a
dispatch and the gradient of a dispatch is a combine, on the forward's
handle.  Review thread: the combine sums rows but does not weight them, so
the routing weights are applied to each expert-output row by the layer (on
the expert's rank, after the expert) and travel with the tokens.

Readings where the page is silent (each one stated here and nowhere else):
  * rank r owns experts [r*E, (r+1)*E), E = e / R;
  * a source sends to each destination the tokens with at least one kept
    route there, in token order (their send slots, rank_slot);
  * a destination receives the arrivals from source 0, then source 1, ...;
  * with each arrival come its k routes' local expert ids (-1 where the
    route goes to another rank or was dropped) and gates;
  * the destination groups its arrivals by local expert in arrival order
    (a dropless layout: no capacity on the receiving side);
  * the partial of an arrival = the fp32 sum, in route order, of gate times
    the expert output over its routes to this rank, rounded once to the
    payload type (the weighted reduction on the expert's rank);
  * the source's output = the fp32 sum, in destination-rank order, of the
    partials it gets back, rounded once;
  * backward: the combine's gradient is sent out like the tokens (a copy
    per destination), the expert rank computes dY and the gate gradients of
    its routes and returns each arrival's gate gradients; the dispatch's
    gradient comes back like the partials and is summed in rank order.
"""
from __future__ import annotations

import numpy as np

from . import combine, combine_bwd, dispatch, dispatch_bwd, layout


def _f32(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def send_plan(idx: np.ndarray, e: int, R: int, capacity: int = 0) -> dict:
    """One source rank's side of the exchange: its layout over R virtual
    ranks, the token-order send slots, and send_row[t, r] = the row of token
    t in the send buffer (destination segments in rank order), -1 where t
    sends nothing to r."""
    L = layout(idx, e, capacity, R)
    counts = L["rank_counts"].astype(np.int64)
    off = np.concatenate([[0], np.cumsum(counts)])
    slot = L["rank_slot"]
    send_row = np.where(slot >= 0, off[:-1][None, :] + slot, -1).astype(np.int32)
    return dict(L=L, rank_counts=counts, send_off=off, send_row=send_row, rows_sent=int(off[-1]))


def send_meta(plan: dict, idx: np.ndarray, gate: np.ndarray, e: int, R: int):
    """For every sent row: the token's k routes as local expert ids on that
    destination (-1: another rank, or dropped) and their gates (0 there)."""
    E = e // R
    s, k = idx.shape
    meta_idx = np.full((plan["rows_sent"], k), -1, np.int32)
    meta_gate = np.zeros((plan["rows_sent"], k), np.float32)
    row = plan["L"]["row"]
    for t in range(s):
        for r in range(R):
            q = plan["send_row"][t, r]
            if q < 0:
                continue
            for j in range(k):
                if row[t, j] >= 0 and idx[t, j] // E == r:
                    meta_idx[q, j] = idx[t, j] - r * E
                    meta_gate[q, j] = gate[t, j]
    return meta_idx, meta_gate


def exchange(bufs: list, counts: np.ndarray) -> list:
    """All-to-all: bufs[src] holds, in destination order, counts[src, dst]
    rows for each destination; returns for every dst the rows from src 0,
    then src 1, ..."""
    R = len(bufs)
    off = [np.concatenate([[0], np.cumsum(counts[src])]) for src in range(R)]
    return [np.concatenate([bufs[src][off[src][dst]:off[src][dst + 1]] for src in range(R)], axis=0)
            for dst in range(R)]


def exchange_back(bufs: list, counts: np.ndarray) -> list:
    """The reverse all-to-all: bufs[dst] holds the rows for src 0, src 1, ...
    (counts[src, dst] each); returns for every src its rows in destination
    order, at the positions it sent them from."""
    return exchange(bufs, counts.T.copy())


def recv_layout(meta_idx: np.ndarray, E: int) -> dict:
    """The receiving rank's layout of its arrivals over its E experts, in
    arrival order, absent routes skipped.  Written with the C layout: an
    absent route j is sent to a sink expert E + j, after every real one, so
    the real experts' slots and offsets are those of the arrivals' real
    routes alone; the sink routes are then dropped (row -1)."""
    n, k = meta_idx.shape
    ids = np.where(meta_idx >= 0, meta_idx, E + np.arange(k, dtype=np.int32)[None, :]).astype(np.int32)
    Lx = layout(ids, E + k, 0, 0)
    row = np.where(meta_idx >= 0, Lx["row"], -1).astype(np.int32)
    return dict(row=row, counts=Lx["counts"][:E].copy(), offsets=Lx["offsets"][:E + 1].copy(),
                rows=int(Lx["offsets"][E]))


def ep_dispatch(xs: list, idxs: list, gates: list, e: int, R: int, capacity: int = 0) -> dict:
    """Every rank's tokens out, every rank's arrivals grouped by local expert.
    xs[r] [s_r, m] (float32, or bf16 as uint16), idxs[r] / gates[r] [s_r, k]."""
    E = e // R
    plans = [send_plan(idxs[r], e, R, capacity) for r in range(R)]
    counts = np.stack([p["rank_counts"] for p in plans])  # [src, dst]
    sends = [dispatch(p["send_row"], xs[r], p["rows_sent"]) for r, p in enumerate(plans)]
    metas = [send_meta(p, idxs[r], gates[r], e, R) for r, p in enumerate(plans)]
    recv_x = exchange(sends, counts)
    recv_idx = exchange([m[0] for m in metas], counts)
    recv_gate = exchange([m[1] for m in metas], counts)
    locs = [recv_layout(recv_idx[d], E) for d in range(R)]
    X = [dispatch(locs[d]["row"], recv_x[d], locs[d]["rows"]) for d in range(R)]
    return dict(E=E, R=R, plans=plans, counts=counts, recv_x=recv_x, recv_idx=recv_idx, recv_gate=recv_gate,
                locs=locs, X=X, idxs=idxs)


def ep_combine(st: dict, ys: list) -> list:
    """ys[d] [rows_d, m]: rank d's expert outputs on its grouped rows.  Each
    arrival's weighted partial on its expert rank, returned to the source
    and summed over destination ranks in rank order."""
    R = st["R"]
    partial = [combine(st["locs"][d]["row"], st["recv_gate"][d], ys[d]) for d in range(R)]
    back = exchange_back(partial, st["counts"])
    return [combine(st["plans"][r]["send_row"], None, back[r]) for r in range(R)]


def ep_combine_bwd(st: dict, douts: list, ys: list):
    """Gradient of ep_combine: (dY[d] per rank's grouped rows, dgate[r] per
    source's routes)."""
    R, E = st["R"], st["E"]
    sends = [dispatch(st["plans"][r]["send_row"], douts[r], st["plans"][r]["rows_sent"]) for r in range(R)]
    recv = exchange(sends, st["counts"])
    dY, dg_recv = [], []
    for d in range(R):
        a, b = combine_bwd(st["locs"][d]["row"], st["recv_gate"][d], recv[d], ys[d])
        dY.append(a)
        dg_recv.append(b)
    dg_back = exchange_back(dg_recv, st["counts"])
    dgate = []
    for r in range(R):
        idx = st["idxs"][r]
        p = st["plans"][r]
        s, k = idx.shape
        g = np.zeros((s, k), np.float32)
        for t in range(s):
            for j in range(k):
                if p["L"]["row"][t, j] >= 0:
                    g[t, j] = dg_back[r][p["send_row"][t, idx[t, j] // E], j]
        dgate.append(g)
    return dY, dgate


def ep_dispatch_bwd(st: dict, dXs: list) -> list:
    """Gradient of ep_dispatch: each arrival's rows summed on its expert
    rank, returned, and summed over destination ranks in rank order."""
    R = st["R"]
    part = [dispatch_bwd(st["locs"][d]["row"], dXs[d]) for d in range(R)]
    back = exchange_back(part, st["counts"])
    return [dispatch_bwd(st["plans"][r]["send_row"], back[r]) for r in range(R)]
