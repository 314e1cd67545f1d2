"""The expert-parallel exchange's host side on real process groups, without
a GPU: gloo ranks (world sizes 2 and 4) exchange counts and rows with the
library's plan and all-to-all (combine_moe_topk_gb300/ep.py), each rank's
local steps taken by the oracle on CPU, and every rank's output, input
gradient and gate gradients must equal the single-process oracle of all
ranks together (oracle/ep.py), bit for bit.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all": the sizes every rank uses must agree (review thread) and the
rows of a combine must be the ones the handle describes.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle import ep as OEP
from combine_moe_topk_gb300 import ep as EP
from combine_moe_topk_gb300 import workloads as W


def rank_inputs(R, s, m, e, k, seed):
    out = []
    for r in range(R):
        w = W.Workload("ep", s=s, m=m, e=e, k=k, dtype="f32", capacity=0, R=R, seed=seed + r, zipf_alpha=1.0)
        inp = W.make_inputs(w)
        idx, gate = oracle.topk_gate(inp["logits"].numpy(), k, 1)
        out.append((inp["x"].numpy(), idx, gate, inp["dout"].numpy()))
    return out


def expert(X, offsets, counts, base):
    ex = np.full(X.shape[0], -1, np.int64)
    for x in range(len(counts)):
        ex[offsets[x]:offsets[x] + counts[x]] = x
    return (X * (np.float32(2.0) ** (((ex + base) % 3) - 1).astype(np.float32))[:, None]).astype(np.float32)


def _rank_main(rank, R, port, args, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=R)
    try:
        s, m, e, k, seed = args
        E = e // R
        x, idx, gate, dout = rank_inputs(R, s, m, e, k, seed)[rank]
        t = torch.from_numpy
        # source: the layout's counts sized by one all-to-all, the send map
        sp = OEP.send_plan(idx, e, R)
        per_dst = np.array([sum(1 for tt in range(s) for j in range(k) if idx[tt, j] // E == d) for d in range(R)])
        plan = EP.exchange_counts(t(sp["rank_counts"].astype(np.int32)), routes=t(per_dst.astype(np.int32)))
        assert plan.rows_sent == sp["rows_sent"]
        mi, mg = OEP.send_meta(sp, idx, gate, e, R)
        rows = EP.all_to_all(t(oracle.dispatch(sp["send_row"], x, sp["rows_sent"])), plan).numpy()
        ids = EP.all_to_all(t(mi), plan).numpy()
        gts = EP.all_to_all(t(mg), plan).numpy()
        assert len(rows) == plan.rows_recv
        # destination: the arrivals grouped, the expert, the weighted partials
        loc = OEP.recv_layout(ids, E)
        assert loc["rows"] == plan.routes_recv  # the exchanged route counts size the grouped rows exactly
        X = oracle.dispatch(loc["row"], rows, loc["rows"])
        y = expert(X, loc["offsets"], loc["counts"], rank * E)
        P = oracle.combine(loc["row"], gts, y)
        out = oracle.combine(sp["send_row"], None, EP.all_to_all(t(P), plan, back=True).numpy())
        # backward
        dP = EP.all_to_all(t(oracle.dispatch(sp["send_row"], dout, sp["rows_sent"])), plan).numpy()
        dY, dg = oracle.combine_bwd(loc["row"], gts, dP, y)
        dg_back = EP.all_to_all(t(dg), plan, back=True).numpy()
        dgate = np.zeros_like(gate)
        for tt in range(s):
            for j in range(k):
                dgate[tt, j] = dg_back[sp["send_row"][tt, idx[tt, j] // E], j]
        dx = oracle.combine(sp["send_row"], None,
                            EP.all_to_all(t(oracle.dispatch_bwd(loc["row"], dY)), plan, back=True).numpy())
        q.put((rank, out, dx, dgate, plan.send_counts, plan.recv_counts))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("R", [2, 4])
def test_gloo_ranks_match_the_single_process_oracle(R):
    s, m, e, k, seed = 120, 8, 16, 4, 50
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + (os.getpid() + R) % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, R, port, (s, m, e, k, seed), q)) for r in range(R)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        r, *vals = q.get(timeout=300)
        got[r] = vals
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inputs = rank_inputs(R, s, m, e, k, seed)
    st = OEP.ep_dispatch([i[0] for i in inputs], [i[1] for i in inputs], [i[2] for i in inputs], e, R)
    E = e // R
    ys = [expert(st["X"][d], st["locs"][d]["offsets"], st["locs"][d]["counts"], d * E) for d in range(R)]
    out = OEP.ep_combine(st, ys)
    dY, dgate = OEP.ep_combine_bwd(st, [i[3] for i in inputs], ys)
    dx = OEP.ep_dispatch_bwd(st, dY)
    for r in range(R):
        o, x_, g, send_counts, recv_counts = got[r]
        assert send_counts == [int(v) for v in st["counts"][r]]
        assert recv_counts == [int(v) for v in st["counts"][:, r]]
        np.testing.assert_array_equal(o, out[r])
        np.testing.assert_array_equal(x_, dx[r])
        np.testing.assert_array_equal(g, dgate[r])
