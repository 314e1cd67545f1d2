"""The expert-parallel steps on one GPU, against the expert-parallel oracle.

R ranks are emulated in one process: each rank's kernels run on its own
tensors, and the all-to-all between them is a permutation of device
tensors done by the test (no kernel waits on another rank's kernel).  Every
rank's outputs -- send map and metadata, arrivals, their layout and grouped
rows, partials, the reduced output, and the backward's dY, gate gradients
and input gradients -- are compared with ``oracle/ep.py`` on the same inputs
(DeepSpeed #8213, description and review thread).
"""
import numpy as np
import pytest
import torch

from oracle import combine as oracle_combine
from oracle import combine_bwd as oracle_combine_bwd
from oracle import dispatch as oracle_dispatch
from oracle import ep as OEP
from oracle import tolerance as T
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import ep as EP
from combine_moe_topk_gb300 import workloads as W
from gpu_util import bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def emulated_all_to_all(bufs, plans, back=False):
    """bufs[i] is rank i's send tensor; returns each rank's receive tensor."""
    R = len(bufs)
    if not back:
        pieces = [torch.split(bufs[src], plans[src].send_counts) for src in range(R)]
        return [torch.cat([pieces[src][dst] for src in range(R)]) for dst in range(R)]
    pieces = [torch.split(bufs[dst], plans[dst].recv_counts) for dst in range(R)]
    return [torch.cat([pieces[dst][src] for dst in range(R)]) for src in range(R)]


def expert_gpu(X, h, base):
    """The test's expert: row times 2^((x % 3) - 1), x = the row's global
    expert (base + its local one); exact in bf16 and fp32."""
    off = h.offsets().long()
    r = torch.arange(X.shape[0], device=X.device)
    x = torch.searchsorted(off, r, right=True) - 1 + base
    return (X.float() * torch.pow(2.0, (x % 3).float() - 1.0)[:, None]).to(X.dtype)


def expert_np(X, offsets, counts, base):
    ex = np.full(X.shape[0], -1, np.int64)
    for x in range(len(counts)):
        ex[offsets[x]:offsets[x] + counts[x]] = x
    scale = np.float32(2.0) ** (((ex + base) % 3) - 1).astype(np.float32)
    if X.dtype == np.uint16:
        f = (X.astype(np.uint32) << 16).view(np.float32) * scale[:, None]
        return (f.view(np.uint32) >> 16).astype(np.uint16)
    return (X * scale[:, None]).astype(np.float32)


def run_case(R, s, m, e, k, dtype, capacity=0, seed=0, zipf=0.0, skip_rank=None):
    """Every step of every rank against the oracle on the same inputs (the
    GPU's own inputs to that step): integers, copies and metadata bit for
    bit, sums within the tolerance rules."""
    E = e // R
    ws = [W.Workload("ep", s=s, m=m, e=e, k=k, dtype=dtype, capacity=capacity, R=R, seed=seed + r, zipf_alpha=zipf)
          for r in range(R)]
    inps = [W.make_inputs(w) for w in ws]
    idx, gate = [], []
    for r in range(R):
        lg = inps[r]["logits"].clone()
        if skip_rank is not None:  # nobody routes to one rank: its segments are empty
            lg[:, skip_rank * E:(skip_rank + 1) * E] = -1e4
        i, g = B.moe_topk_gate(lg.to(DEV), k, 1)
        idx.append(i)
        gate.append(g)
    xs = [inps[r]["x"].to(DEV) for r in range(R)]
    douts = [inps[r]["dout"].to(DEV) for r in range(R)]
    # ---- forward, rank by rank with the exchange between the phases
    hs = [B.moe_dispatch_layout_ex(idx[r], e, capacity, R, send_slots=True) for r in range(R)]
    counts = torch.stack([h.rank_counts() for h in hs]).cpu().numpy().astype(np.int64)  # [src, dst]
    routes = torch.stack([EP.route_counts(h) for h in hs]).cpu().numpy().astype(np.int64)  # [src, dst]
    plans = [EP.Plan(send_counts=[int(v) for v in counts[r]], recv_counts=[int(v) for v in counts[:, r]],
                     recv_routes=[int(v) for v in routes[:, r]]) for r in range(R)]
    sends = [EP.source_send(hs[r], xs[r], gate[r], plans[r]) for r in range(R)]
    rows = emulated_all_to_all([sd.X_send for sd in sends], plans)
    ids = emulated_all_to_all([sd.meta_idx for sd in sends], plans)
    gts = emulated_all_to_all([sd.meta_gate for sd in sends], plans)
    # the grouped buffers sized exactly by the exchanged route counts
    recvs = [EP.dest_receive(rows[d], ids[d], gts[d], E, plans[d].routes_recv) for d in range(R)]
    ys = [expert_gpu(recvs[d].X, recvs[d].h, d * E) for d in range(R)]
    P = [EP.dest_partial(recvs[d], ys[d]) for d in range(R)]
    P_back = emulated_all_to_all(P, plans, back=True)
    outs = [EP.source_reduce(hs[r], sends[r], P_back[r]) for r in range(R)]
    # ---- backward
    dP = emulated_all_to_all([EP.source_send_grad(hs[r], sends[r], douts[r]) for r in range(R)], plans)
    cb = [EP.dest_combine_bwd(recvs[d], dP[d], ys[d]) for d in range(R)]
    dgb = emulated_all_to_all([c[1] for c in cb], plans, back=True)
    dgates = [EP.source_dgate(hs[r], sends[r], dgb[r]) for r in range(R)]
    dxp = [EP.dest_dispatch_bwd(recvs[d], cb[d][0]) for d in range(R)]
    dxb = emulated_all_to_all(dxp, plans, back=True)
    dxs = [EP.source_reduce(hs[r], sends[r], dxb[r]) for r in range(R)]
    torch.cuda.synchronize()
    for h in hs + [rc.h for rc in recvs]:
        assert h.status() == 0

    # ---- the oracle
    oi = [bits(i) for i in idx]
    og = [bits(g) for g in gate]
    st = OEP.ep_dispatch([bits(x) for x in xs], oi, og, e, R, capacity)
    np.testing.assert_array_equal(counts, st["counts"])
    for r in range(R):
        srow = st["plans"][r]["send_row"]
        np.testing.assert_array_equal(bits(sends[r].send_row), srow, err_msg="send_row")
        mi, mg = OEP.send_meta(st["plans"][r], oi[r], og[r], e, R)
        np.testing.assert_array_equal(bits(sends[r].meta_idx), mi, err_msg="meta_idx")
        np.testing.assert_array_equal(bits(sends[r].meta_gate), mg, err_msg="meta_gate")
    for d in range(R):
        loc = st["locs"][d]
        lr = loc["row"]
        np.testing.assert_array_equal(bits(rows[d]), st["recv_x"][d], err_msg="arrivals")
        np.testing.assert_array_equal(bits(gts[d]), st["recv_gate"][d], err_msg="arrivals' gates")
        np.testing.assert_array_equal(bits(recvs[d].h.row()), lr, err_msg="arrivals' rows")
        np.testing.assert_array_equal(bits(recvs[d].h.counts()), loc["counts"], err_msg="arrivals' counts")
        np.testing.assert_array_equal(bits(recvs[d].h.offsets()), loc["offsets"], err_msg="arrivals' offsets")
        lrows = loc["rows"]
        assert recvs[d].h.rows == lrows == plans[d].routes_recv  # sized exactly from the exchanged counts
        X = bits(recvs[d].X)[:lrows]
        np.testing.assert_array_equal(X, st["X"][d], err_msg="grouped rows")
        y = bits(ys[d])[:lrows]
        np.testing.assert_array_equal(y, expert_np(st["X"][d], loc["offsets"], loc["counts"], d * E))
        g = st["recv_gate"][d]
        T.assert_close(bits(P[d]), oracle_combine(lr, g, y), T.combine_scale(lr, g, y), "partial")
        dPd = bits(dP[d])
        np.testing.assert_array_equal(dPd, OEP.exchange(
            [oracle_dispatch(st["plans"][r]["send_row"], bits(douts[r]), st["plans"][r]["rows_sent"])
             for r in range(R)], st["counts"])[d], err_msg="outgoing gradient")
        OdY, Odg = oracle_combine_bwd(lr, g, dPd, y)
        T.assert_close(bits(cb[d][0])[:lrows], OdY, np.abs(T.as_f64(OdY)), "dY")
        T.assert_close(bits(cb[d][1]), Odg, T.dot_scale(lr, dPd, y), "arrivals' dgate")
        dYd = bits(cb[d][0])[:lrows]
        T.assert_close(bits(dxp[d]), oracle_combine(lr, None, dYd), T.combine_scale(lr, None, dYd), "dx partial")
    for r in range(R):
        srow = st["plans"][r]["send_row"]
        pb = bits(P_back[r])
        T.assert_close(bits(outs[r]), oracle_combine(srow, None, pb), T.combine_scale(srow, None, pb), "out")
        xb = bits(dxb[r])
        T.assert_close(bits(dxs[r]), oracle_combine(srow, None, xb), T.combine_scale(srow, None, xb), "dx")
        # the gate gradients returned, gathered back to the source's routes
        want = np.zeros((s, k), np.float32)
        row = st["plans"][r]["L"]["row"]
        got_back = bits(dgb[r])
        for t in range(s):
            for j in range(k):
                if row[t, j] >= 0:
                    want[t, j] = got_back[srow[t, oi[r][t, j] // E], j]
        np.testing.assert_array_equal(bits(dgates[r]), want, err_msg="dgate")
    return st


@pytest.mark.parametrize("case", [
    dict(R=2, s=300, m=64, e=8, k=2, dtype="f32"),
    dict(R=4, s=1000, m=128, e=16, k=4, dtype="bf16", zipf=1.0),
    dict(R=8, s=777, m=64, e=64, k=8, dtype="bf16", zipf=1.5),
    dict(R=8, s=500, m=32, e=16, k=6, dtype="f32"),                   # E = 2 < k: more routes than local experts
    dict(R=4, s=600, m=64, e=32, k=4, dtype="bf16", capacity=40),     # capacity drops are not sent
    dict(R=4, s=400, m=64, e=16, k=2, dtype="bf16", skip_rank=2),     # a rank nobody sends to
    dict(R=1, s=256, m=64, e=8, k=2, dtype="f32"),                    # one rank: the one-GPU path
    dict(R=16, s=300, m=32, e=64, k=5, dtype="bf16"),
    dict(R=32, s=200, m=32, e=64, k=4, dtype="f32"),
], ids=lambda c: "-".join(f"{k_}{v}" for k_, v in c.items()))
def test_expert_parallel_against_the_oracle(case):
    run_case(**case)


def test_expert_parallel_fine_grained_routing():
    """The fine-grained skewed routing (128 experts, top-8, the Zipf-like
    bias) over 8 ranks of 16 experts, 4096 tokens per rank."""
    st = run_case(R=8, s=4096, m=64, e=128, k=8, dtype="bf16", zipf=1.5, seed=3)
    # dedup: fewer rows cross than routes exist
    assert int(st["counts"].sum()) < 8 * 4096 * 8


def test_ep_calls_reject_a_handle_without_send_slots():
    idx = W.random_routes(64, 8, 2, device=DEV)
    h = B.moe_dispatch_layout_ex(idx, 8, 0, 2)
    with pytest.raises(B.MoEError) as ei:
        B.moe_ep_pack(h, torch.ones(64, 2, device=DEV), 10)
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    hs = B.moe_dispatch_layout_ex(idx, 8, 0, 2, send_slots=True)
    with pytest.raises(B.MoEError):
        B.moe_ep_pack(hs, torch.ones(64, 2, device=DEV), 64 * 2 + 1)  # more rows than s*R


def test_expert_parallel_layer_on_a_one_rank_group():
    """ExpertParallelMoE end to end over a real (one-rank, NCCL) process
    group: with one rank it must give the one-GPU path's bits -- forward,
    input gradient and gate gradients."""
    import socket

    import torch.distributed as dist

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=DEV)
    try:
        w = W.Workload("ep1", s=700, m=128, e=16, k=4, dtype="bf16", capacity=0, R=1, seed=21)
        inp = W.make_inputs(w, device=DEV)
        idx, gate = B.moe_topk_gate(inp["logits"], w.k, 1)
        layer = EP.ExpertParallelMoE(w.e)
        assert (layer.R, layer.E) == (1, 16)
        h, plan = layer.layout(idx)
        assert plan.rows_sent == plan.rows_recv == w.s
        fwd = lambda recv: expert_gpu(recv.X, recv.h, 0)
        bwd = lambda recv, dY: expert_gpu(dY, recv.h, 0)  # the expert is a per-expert scale: its own adjoint
        out, saved = layer.forward(h, plan, inp["x"], gate, fwd)
        dx, dgate = layer.backward(h, plan, saved, inp["dout"], bwd)
        # the one-GPU path on the same routes
        h1 = B.moe_dispatch_layout(idx, w.e)
        X = B.moe_dispatch(h1, inp["x"])
        y = expert_gpu(X, h1, 0)
        ref = B.moe_combine(h1, y, gate)
        dY, dg = B.moe_combine_bwd(h1, inp["dout"], gate, y)
        dxr = B.moe_dispatch_bwd(h1, expert_gpu(dY, h1, 0))
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(dx, dxr)
        assert torch.equal(dgate.view(torch.int32), dg.view(torch.int32))
    finally:
        dist.destroy_process_group()


def test_rows_bound_below_the_routes_cuts_and_reports():
    """A dropless bound smaller than the routes: the routes past it get no
    row, the segments are cut at the bound, the status says so, and the
    dispatch writes nothing past the buffer."""
    s, e, k = 500, 8, 2
    idx = W.random_routes(s, e, k, device=DEV, seed=4)
    bound = s * k - 137
    h = B.moe_dispatch_layout_ex(idx, e, rows_bound=bound)
    assert h.rows == bound
    assert h.status() & B.MOE_DEV_ROWS_EXCEEDED
    L = __import__("oracle").layout(bits(idx), e)
    row = bits(h.row())
    full = L["row"]
    np.testing.assert_array_equal(row, np.where(full < bound, full, -1))
    off = bits(h.offsets())
    cnt = bits(h.counts())
    assert off[-1] == bound and np.all(off[:-1] + cnt <= bound)
    np.testing.assert_array_equal(off, np.minimum(L["offsets"], bound))
    x = torch.randn(s, 16, device=DEV)
    guard = torch.full((bound + 64, 16), 7.0, device=DEV)
    B.moe_dispatch(h, x, guard[:bound])
    torch.cuda.synchronize()
    assert torch.all(guard[bound:] == 7.0)  # nothing past the rows
    exact = B.moe_dispatch_layout_ex(idx, e, rows_bound=s * k)
    assert exact.status() == 0 and exact.rows == s * k
