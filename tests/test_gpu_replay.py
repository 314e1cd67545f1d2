"""Activation-checkpoint replay on cached handles, and the autograd wrappers.

Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
activation-checkpoint recompute": 30 layers x 3 passes need 90 dispatches;
activation checkpointing replays the encoder and the real-decode passes
(60 replays), each of which must reuse the logged handle -- no layout
rebuild -- and reproduce bit-identical counts and outputs; the top-k index
checksum of a recompute equals the forward's.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as T
from combine_moe_topk_gb300 import autograd as A
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W
from gpu_util import bits, check_layout, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_stacked_replay_90_builds_60_replays():
    w = W.WORKLOADS["diffusiongemma-replay"]
    replayed_passes = (0, 2)  # the checkpointed passes; pass 1 runs without grad
    recorders = {}
    fwd = {}
    n_builds = 0
    for p in range(w.passes):
        for layer in range(w.layers):
            inp = W.make_inputs(w, device=DEV, seed=W.replay_seed(w, p, layer), with_grad=False)
            idx, gate = B.moe_topk_gate(inp["logits"], w.k)
            rec = A.HandleRecorder(verify=True) if p in replayed_passes else None
            h = rec.layout(idx, w.e) if rec is not None else B.moe_dispatch_layout(idx, w.e)
            n_builds += 1
            X = B.moe_dispatch(h, inp["x"])
            out = B.moe_combine(h, X, gate)  # identity expert
            if rec is not None:
                recorders[(p, layer)] = rec
                fwd[(p, layer)] = (int(idx.sum()), bits(h.counts()), bits(h.offsets()), X, out)
            if p == 1 and layer == 0:
                # one sampled build checked against the oracle in full
                oi, og = oracle.topk_gate(bits(inp["logits"]), w.k)
                np.testing.assert_array_equal(bits(idx), oi)
                check_layout(h, oracle.layout(oi, w.e), oi)
    assert n_builds == 90

    layouts = B.moe_launch_count("layout")
    n_replays = 0
    for p in reversed(replayed_passes):          # backward runs the later pass first
        for layer in reversed(range(w.layers)):  # and the layers in reverse
            inp = W.make_inputs(w, device=DEV, seed=W.replay_seed(w, p, layer), with_grad=False)
            idx, gate = B.moe_topk_gate(inp["logits"], w.k)  # routing pinned: recomputed identically
            rec = recorders[(p, layer)].replay()
            h = rec.layout(idx, w.e)
            X = B.moe_dispatch(h, inp["x"])
            out = B.moe_combine(h, X, gate)
            checksum, counts, offsets, X0, out0 = fwd[(p, layer)]
            assert int(idx.sum()) == checksum
            np.testing.assert_array_equal(bits(h.counts()), counts)
            np.testing.assert_array_equal(bits(h.offsets()), offsets)
            assert torch.equal(X, X0) and torch.equal(out, out0)
            assert rec.replayed == 1 and rec.fallbacks == 0
            n_replays += 1
    assert n_replays == 60
    assert B.moe_launch_count("layout") == layouts, "a replay must not launch the layout kernel"


def test_recorder_outrun_rebuilds_on_gpu():
    w = W.WORKLOADS["diffusiongemma-replay"].replace(m=256)
    inp = W.make_inputs(w, device=DEV, with_grad=False)
    idx, _ = B.moe_topk_gate(inp["logits"], w.k)
    rec = A.HandleRecorder()
    h0 = rec.layout(idx, w.e)
    rec.replay()
    n = B.moe_launch_count("layout")
    assert rec.layout(idx, w.e) is h0 and B.moe_launch_count("layout") == n
    h1 = rec.layout(idx, w.e)  # log exhausted: a fresh, correct build
    assert h1 is not h0 and B.moe_launch_count("layout") == n + 1 and rec.fallbacks == 1
    assert torch.equal(h1.row(), h0.row())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("capacity", [0, 150])
def test_autograd_matches_oracle(dtype, capacity):
    """loss = <combine(2 * dispatch(x), gate), dout>: x.grad and gate.grad from
    torch.autograd through the library's backward entry points."""
    s, m, e, k = 700, 64, 16, 4
    w = W.Workload("autograd", s=s, m=m, e=e, k=k, dtype=dtype, capacity=capacity, R=0, seed=31)
    inp = W.make_inputs(w)
    oi, og = oracle.topk_gate(inp["logits"].numpy(), k)
    L = oracle.layout(oi, e, capacity)
    h = B.moe_dispatch_layout(to_dev(oi, DEV), e, capacity)

    x = inp["x"].to(DEV).requires_grad_(True)
    gate = to_dev(og, DEV).requires_grad_(True)
    X = A.dispatch(x, h)
    y = X * 2
    out = A.combine(y, gate, h)
    dout = inp["dout"].to(DEV)
    out.backward(dout)

    xb, db = bits(inp["x"]), bits(inp["dout"])
    OX = oracle.dispatch(L["row"], xb, L["rows"])
    np.testing.assert_array_equal(bits(X), OX)
    Oy = (T.as_f64(OX) * 2).astype(np.float32)
    if dtype == "bf16":
        Oy = bits(torch.from_numpy(Oy).to(torch.bfloat16))  # exact: doubling a bf16 value
    OdY, Odg = oracle.combine_bwd(L["row"], og, db, Oy)
    T.assert_close(bits(gate.grad), Odg, T.dot_scale(L["row"], db, Oy), "gate.grad")
    OdX = (T.as_f64(OdY) * 2).astype(np.float32)
    if dtype == "bf16":
        OdX = bits(torch.from_numpy(OdX).to(torch.bfloat16))
    Odx = oracle.dispatch_bwd(L["row"], OdX)
    T.assert_close(bits(x.grad), Odx, T.combine_scale(L["row"], None, OdX), "x.grad")


@pytest.mark.parametrize("renorm", [0, 1])
def test_router_gradient_through_the_whole_path(renorm):
    """logits -> top-k gate -> layout -> dispatch -> expert (2x) -> combine ->
    loss; torch.autograd reaches the logits through moe_topk_gate_bwd.  Each op
    is held to its own bar elsewhere; here the chain (GPU gates feed the GPU
    ops) is compared with the oracle's chain within 1e-5 of the scale."""
    s, m, e, k = 600, 64, 32, 4
    w = W.Workload("chain", s=s, m=m, e=e, k=k, dtype="f32", capacity=0, R=0, seed=41)
    inp = W.make_inputs(w)
    logits = inp["logits"].to(DEV).requires_grad_(True)
    idx, gate = A.topk_gate(logits, k, renorm)
    h = B.moe_dispatch_layout(idx, e)
    X = A.dispatch(inp["x"].to(DEV), h)
    out = A.combine(X * 2, gate, h)
    dout = inp["dout"].to(DEV)
    out.backward(dout)

    lg = inp["logits"].numpy()
    oi, og = oracle.topk_gate(lg, k, renorm)
    np.testing.assert_array_equal(bits(idx), oi)
    L = oracle.layout(oi, e)
    Oy = (oracle.dispatch(L["row"], inp["x"].numpy(), L["rows"]) * 2).astype(np.float32)
    _, Odg = oracle.combine_bwd(L["row"], og, inp["dout"].numpy(), Oy)
    Odl = oracle.topk_gate_bwd(lg, oi, og, Odg, e, renorm)
    got = bits(logits.grad)
    # the upstream gate gradient carries its own fp32 error, on the scale sum |dout * y|
    scale = T.gate_bwd_scale(oi, og, T.dot_scale(L["row"], inp["dout"].numpy(), Oy), e, renorm, lg)
    bad = np.abs(got.astype(np.float64) - Odl) > 1e-5 * scale + 1e-30
    assert not bad.any(), (int(bad.sum()), np.abs(got - Odl).max())


def test_recorder_replays_layout_variants():
    """k-major capacity priority and padded dropless layouts (with send
    slots) replay through the recorder like plain ones: no layout launch,
    identical rows and slots."""
    idx = W.random_routes(3000, 32, 4, device=DEV, seed=23)
    rec = A.HandleRecorder(verify=True)
    h1 = rec.layout(idx, 32, 300, 4, priority="kmajor")
    h2 = rec.layout(idx, 32, 0, 4, pad_multiple=128, send_slots=True)
    rows1, rows2, slots2 = h1.row().clone(), h2.row().clone(), h2.rank_slot().clone()
    rec.replay()
    n = B.moe_launch_count("layout")
    r1 = rec.layout(idx, 32, 300, 4, priority="kmajor")
    r2 = rec.layout(idx, 32, 0, 4, pad_multiple=128, send_slots=True)
    assert r1 is h1 and r2 is h2 and B.moe_launch_count("layout") == n
    assert torch.equal(r1.row(), rows1) and torch.equal(r2.row(), rows2) and torch.equal(r2.rank_slot(), slots2)
    assert r1.priority == 1 and r2.pad_multiple == 128
