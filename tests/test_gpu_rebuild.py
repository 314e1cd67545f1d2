"""Layouts built in place: a handle created once and rebuilt from new routes
(no allocation, no memset), and the top-k gate fused into the layout build.

Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
activation-checkpoint recompute", description: the layout is recomputed
every step, so its per-step cost matters.  Every rebuild must give exactly
the layout a fresh build gives (bit-exact against the oracle), whatever the
previous build left in the handle's memory.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as T
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W
from gpu_util import bits, check_layout, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

SHAPES = {
    "tiny-capacity": W.WORKLOADS["tiny-capacity"],
    "mixtral-dropless": W.WORKLOADS["mixtral-dropless"].replace(m=256),
    "fine-grained-skewed": W.WORKLOADS["fine-grained-skewed"].replace(m=256),
    "diffusiongemma-replay": W.WORKLOADS["diffusiongemma-replay"].replace(m=256),
    "gshard-capacity": W.WORKLOADS["gshard-capacity"].replace(m=128),
}


def _oracle_layout(ids, w, priority=0, pad=1):
    return oracle.layout(ids, w.e, w.capacity, w.R, priority=priority, pad_multiple=pad)


@pytest.mark.parametrize("name", list(SHAPES))
def test_rebuilds_match_the_oracle_every_time(name):
    """One handle, five builds from different routes (alternating look-back
    parity), each bit-exact against the oracle; the status word and the rank
    counts start from zero on every build."""
    w = SHAPES[name]
    h = B.moe_layout_create(w.s, w.e, w.k, w.capacity, w.R, device=DEV)
    for seed in range(5):
        ids = oracle.topk_gate(W.make_logits(w, seed=100 + seed).numpy(), w.k, w.renorm)[0]
        B.moe_layout_rebuild(h, to_dev(ids, DEV))
        check_layout(h, _oracle_layout(ids, w), ids)
        assert h.status() == 0
    h.destroy()


@pytest.mark.parametrize("variant", [dict(priority="kmajor"), dict(pad_multiple=8), dict(send_slots=True)],
                         ids=["kmajor", "padded", "send-slots"])
def test_rebuilds_of_layout_variants(variant):
    w = SHAPES["gshard-capacity"] if "priority" in variant else SHAPES["fine-grained-skewed"]
    if "pad_multiple" in variant:
        w = w.replace(capacity=0)
    h = B.moe_layout_create(w.s, w.e, w.k, w.capacity, w.R, device=DEV, **variant)
    for seed in range(3):
        ids = W.random_routes(w.s, w.e, w.k, seed=200 + seed).numpy()
        B.moe_layout_rebuild(h, to_dev(ids, DEV))
        L = _oracle_layout(ids, w, priority=1 if variant.get("priority") == "kmajor" else 0,
                           pad=variant.get("pad_multiple", 1))
        check_layout(h, L, ids)
        if variant.get("send_slots"):
            np.testing.assert_array_equal(bits(h.rank_slot()), L["rank_slot"])
        assert h.status() == 0
    h.destroy()


def test_payload_on_a_rebuilt_handle_follows_the_new_layout():
    """Dispatch and combine enqueued after a rebuild use the new layout."""
    w = SHAPES["mixtral-dropless"]
    inp = W.make_inputs(w)
    h = B.moe_layout_create(w.s, w.e, w.k, device=DEV)
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch(h, inp["x"].to(DEV))  # no layout yet
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    for seed in (1, 2):
        ids = W.random_routes(w.s, w.e, w.k, seed=seed).numpy()
        B.moe_layout_rebuild(h, to_dev(ids, DEV))
        L = _oracle_layout(ids, w)
        X = B.moe_dispatch(h, inp["x"].to(DEV))
        np.testing.assert_array_equal(bits(X), oracle.dispatch(L["row"], bits(inp["x"]), L["rows"]))
    h.destroy()


@pytest.mark.parametrize("renorm", [1, 0])
@pytest.mark.parametrize("name", list(SHAPES))
def test_gate_fused_into_the_layout(name, renorm):
    """moe_topk_gate_layout: ids bit-exact and gates within 1e-6 of the
    oracle, and the same bits as the separate gate kernel; the layout
    bit-exact against the oracle's layout of those ids; twice in a row."""
    w = SHAPES[name].replace(s=W.WORKLOADS[name].s)  # the workload's own token count
    h = B.moe_layout_create(w.s, w.e, w.k, w.capacity, w.R, device=DEV)
    n_fused, n_gate = B.moe_launch_count("gate_layout"), B.moe_launch_count("topk_gate")
    for seed in (w.seed, w.seed + 1):
        logits = W.make_logits(w, seed=seed)
        idx, gate = B.moe_topk_gate_layout(h, logits.to(DEV), renorm)
        oi, og = oracle.topk_gate(logits.numpy(), w.k, renorm)
        np.testing.assert_array_equal(bits(idx), oi)
        T.assert_gates_close(bits(gate), og)
        idx2, gate2 = B.moe_topk_gate(logits.to(DEV), w.k, renorm)
        assert torch.equal(idx, idx2) and torch.equal(gate.view(torch.int32), gate2.view(torch.int32))
        check_layout(h, _oracle_layout(oi, w), oi)
        assert h.status() == 0
    # one kernel up to 32 experts; the gate kernel then the layout beyond
    fused = 2 if w.e <= 32 else 0
    assert B.moe_launch_count("gate_layout") == n_fused + fused
    assert B.moe_launch_count("topk_gate") == n_gate + 4 - fused  # + the two separate calls above
    h.destroy()


@pytest.mark.parametrize("case", [
    dict(s=5000, e=16, k=6, capacity=400, R=4, priority="kmajor"),   # k-major: gate kernel, then layout
    dict(s=1 << 18, e=32, k=4, capacity=0, R=8, priority="token"),   # tiles span four sub-tiles
    dict(s=3001, e=64, k=4, capacity=0, R=0, priority="token"),      # more than 32 experts
], ids=["kmajor", "many-subtiles", "e64"])
def test_gate_layout_where_the_layout_cannot_select(case):
    """Where the layout kernel cannot run the gate itself, the same entry
    point launches the gate kernel and then the layout: the same results."""
    w = W.Workload("gl", s=case["s"], m=8, e=case["e"], k=case["k"], dtype="f32", capacity=case["capacity"],
                   R=case["R"], seed=13)
    h = B.moe_layout_create(w.s, w.e, w.k, w.capacity, w.R, priority=case["priority"], device=DEV)
    n_gate = B.moe_launch_count("topk_gate")
    for seed in (1, 2):
        logits = W.make_logits(w, seed=seed)
        idx, gate = B.moe_topk_gate_layout(h, logits.to(DEV), 1)
        oi, og = oracle.topk_gate(logits.numpy(), w.k, 1)
        np.testing.assert_array_equal(bits(idx), oi)
        T.assert_gates_close(bits(gate), og)
        check_layout(h, _oracle_layout(oi, w, priority=1 if case["priority"] == "kmajor" else 0), oi)
        assert h.status() == 0
    assert B.moe_launch_count("topk_gate") == n_gate + 2
    h.destroy()


@pytest.mark.parametrize("case", [
    dict(s=1000, e=32, k=16), dict(s=777, e=7, k=3), dict(s=300, e=1, k=1), dict(s=513, e=30, k=5),
    # the 8-expert form's edges (k = e; 16-byte rows of 4) and the 32-expert form's smallest e
    dict(s=600, e=8, k=8), dict(s=900, e=4, k=2), dict(s=450, e=9, k=2),
], ids=lambda c: f"e{c['e']}-k{c['k']}")
@pytest.mark.parametrize("renorm", [1, 0])
def test_fused_gate_edges_and_ties(case, renorm):
    """The fused gate's thread-per-token selection at the edges of its range
    (e = 32 with k = 16, odd e without 16-byte rows, e = 1; the 8-expert
    form at k = e and e = 4, the 32-expert form at e = 9), with logits on a
    small grid so that ties are everywhere: the gate kernel's bits."""
    s, e, k = case["s"], case["e"], case["k"]
    g = torch.Generator().manual_seed(e * 100 + k)
    logits = (torch.randint(-3, 4, (s, e), generator=g).float() * 0.5)
    logits[::7] = -logits[::7]  # -0.0 against +0.0 as well
    h = B.moe_layout_create(s, e, k, device=DEV)
    n_fused = B.moe_launch_count("gate_layout")
    idx, gate = B.moe_topk_gate_layout(h, logits.to(DEV), renorm)
    assert B.moe_launch_count("gate_layout") == n_fused + 1
    idx2, gate2 = B.moe_topk_gate(logits.to(DEV), k, renorm)
    assert torch.equal(idx, idx2) and torch.equal(gate.view(torch.int32), gate2.view(torch.int32))
    oi, og = oracle.topk_gate(logits.numpy(), k, renorm)
    np.testing.assert_array_equal(bits(idx), oi)
    T.assert_gates_close(bits(gate), og)
    check_layout(h, oracle.layout(oi, e), oi)
    assert h.status() == 0
    h.destroy()


def test_fused_gate_flags_nonfinite_logits_and_rebuild_clears_it():
    w = SHAPES["mixtral-dropless"].replace(s=700)
    h = B.moe_layout_create(w.s, w.e, w.k, device=DEV)
    logits = W.make_logits(w, device=DEV)
    bad = logits.clone()
    bad[123, 4] = float("nan")
    B.moe_topk_gate_layout(h, bad, 1)
    assert h.status() & B.MOE_DEV_NONFINITE
    B.moe_topk_gate_layout(h, logits, 1)
    assert h.status() == 0


def test_rebuild_after_a_timed_out_build():
    """A build whose look-back wait ran out (one tile held back) still leaves
    every tile's row rewritten, so the next build -- with the other parity --
    is exact and its status clean."""
    s, e, k = 256 * 6, 8, 2
    h = B.moe_layout_create(s, e, k, device=DEV)
    idx = W.random_routes(s, e, k, device=DEV, seed=1)
    B.moe_layout_rebuild(h, idx)
    B.moe_debug_hold_layout_tile(2, timeout_ms=200)
    idx2 = W.random_routes(s, e, k, device=DEV, seed=2)
    B.moe_layout_rebuild(h, idx2)
    assert h.status() & B.MOE_DEV_TIMEOUT
    for seed in (3, 4):
        idx3 = W.random_routes(s, e, k, device=DEV, seed=seed)
        B.moe_layout_rebuild(h, idx3)
        assert h.status() == 0
        check_layout(h, oracle.layout(bits(idx3), e), bits(idx3))
    h.destroy()
