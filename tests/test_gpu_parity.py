"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Reduced sizes run every output of every op element by element, at sizes that
still span several layout tiles (256 tokens each) and end in a ragged tail.
The full workload shapes are compared in full as well: every integer
output, gate, dispatched row and every element of the floating outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as T
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W
from gpu_util import bits, check_layout, full_parity, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

REDUCED = {
    "tiny-capacity": W.WORKLOADS["tiny-capacity"],
    "mixtral-dropless": W.WORKLOADS["mixtral-dropless"].replace(s=1000, m=512),
    "fine-grained-skewed": W.WORKLOADS["fine-grained-skewed"].replace(s=3000, m=256),
    "diffusiongemma-replay": W.WORKLOADS["diffusiongemma-replay"].replace(m=256),
    "gshard-capacity": W.WORKLOADS["gshard-capacity"].replace(s=5000, m=128, capacity=469),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_reduced_full_parity(name):
    full_parity(REDUCED[name], DEV)


@pytest.mark.parametrize("name", ["tiny-capacity", "gshard-capacity", "fine-grained-skewed", "mixtral-dropless"])
def test_kmajor_priority_parity(name):
    """GShard's order: every first choice before any second choice."""
    full_parity(REDUCED[name], DEV, priority="kmajor")


@pytest.mark.parametrize("pad", [4, 128])
@pytest.mark.parametrize("name", ["mixtral-dropless", "fine-grained-skewed", "diffusiongemma-replay"])
def test_padded_grouped_layout_parity(name, pad):
    """Dropless rows padded per expert to a multiple: padding rows are zero."""
    full_parity(REDUCED[name], DEV, pad_multiple=pad)


def test_kmajor_with_padding_and_dedup():
    full_parity(REDUCED["fine-grained-skewed"].replace(s=1500), DEV, priority="kmajor", pad_multiple=8)


@pytest.mark.parametrize("case", [
    dict(s=16384, e=128, k=8, capacity=0, R=8, priority="token"),      # fine-grained shape, full size
    dict(s=32768, e=64, k=6, capacity=3072, R=16, priority="token"),   # GShard shape with drops, full size
    dict(s=5000, e=64, k=6, capacity=400, R=4, priority="kmajor"),
    dict(s=20001, e=128, k=4, capacity=0, R=64, priority="token"),     # two scan chunks, ragged, 64 ranks
    dict(s=3, e=4, k=2, capacity=1, R=2, priority="token"),
], ids=lambda c: f"s{c['s']}-e{c['e']}-R{c['R']}-c{c['capacity']}-{c['priority']}")
def test_send_slots_parity(case):
    """Per-virtual-rank token-order send slots: bit-exact against the oracle,
    and the rest of the layout unchanged by asking for them."""
    idx = W.random_routes(case["s"], case["e"], case["k"], seed=17).numpy()
    h = B.moe_dispatch_layout_ex(to_dev(idx, DEV), case["e"], case["capacity"], case["R"], case["priority"],
                                 send_slots=True)
    L = oracle.layout(idx, case["e"], case["capacity"], case["R"],
                      priority=1 if case["priority"] == "kmajor" else 0)
    check_layout(h, L, idx)
    np.testing.assert_array_equal(bits(h.rank_slot()), L["rank_slot"])
    assert h.status() == 0
    plain = B.moe_dispatch_layout_ex(to_dev(idx, DEV), case["e"], case["capacity"], case["R"], case["priority"])
    with pytest.raises(B.MoEError):
        plain.rank_slot()


def test_tiny_capacity_as_specified_with_the_affine_expert():
    """The tiny capacity workload exactly as specified, forward only: seed-0
    logits [256, 8] and x [256, 128] fp32, capacity ceil(1.25*256*2/8) = 80
    in token order with drops, and the expert output y = 2*X + 1 elementwise
    on the dispatched buffer (formed in fp32 on the host from the oracle's
    X, which the GPU's X equals bit for bit).  Gate, layout, dispatch and
    combine against the oracle, element by element; the combine on the
    GPU's own gates, fed to both sides."""
    w = W.WORKLOADS["tiny-capacity"]
    assert (w.s, w.m, w.e, w.k, w.seed) == (256, 128, 8, 2, 0)
    assert w.capacity == B.moe_capacity(1.25, w.s, w.k, w.e) == 80
    inp = W.make_inputs(w, with_grad=False)
    logits, x = inp["logits"].numpy(), inp["x"].numpy()
    idx, gate = B.moe_topk_gate(inp["logits"].to(DEV), w.k, w.renorm)
    oi, og = oracle.topk_gate(logits, w.k, w.renorm)
    np.testing.assert_array_equal(bits(idx), oi)
    T.assert_gates_close(bits(gate), og)

    h = B.moe_dispatch_layout(idx, w.e, w.capacity)
    L = oracle.layout(oi, w.e, w.capacity)
    check_layout(h, L, oi)
    assert L["drop"].any(), "capacity 80 drops routes on this workload"
    X = B.moe_dispatch(h, inp["x"].to(DEV))
    OX = oracle.dispatch(L["row"], x, L["rows"])
    np.testing.assert_array_equal(bits(X), OX, err_msg="dispatch")

    y = np.float32(2.0) * OX + np.float32(1.0)  # the expert, on every slot (unused slots hold 1, never read)
    g = bits(gate)
    out = B.moe_combine(h, to_dev(y, DEV), gate)
    ref = oracle.combine(L["row"], g, y)
    T.assert_close(bits(out), ref, T.combine_scale(L["row"], g, y), "combine")
    # what the affine expert gives: out[t] = (sum of kept gates) * (2 x[t] + 1)
    kept_g = np.where(L["row"] >= 0, g.astype(np.float64), 0.0).sum(axis=1, keepdims=True)
    expect = kept_g * (2.0 * x.astype(np.float64) + 1.0)
    assert np.all(np.abs(bits(out) - expect) <= 1e-6 * np.abs(kept_g) * np.abs(2.0 * x + 1.0) + 1e-30)
    assert np.all(bits(out)[(L["row"] < 0).all(axis=1)] == 0), "fully dropped tokens give zeros"
    assert h.status() == 0


def test_tiny_capacity_full_softmax_gates():
    full_parity(W.WORKLOADS["tiny-capacity"], DEV, renorm=0)


@pytest.mark.parametrize("case", [
    dict(s=1, m=8, e=1, k=1, dtype="bf16", capacity=0, R=0),
    dict(s=1, m=4, e=4, k=4, dtype="f32", capacity=1, R=2),
    dict(s=37, m=8, e=256, k=16, dtype="bf16", capacity=0, R=64),
    dict(s=300, m=12288, e=16, k=3, dtype="bf16", capacity=0, R=4),   # a short batch: rows split into 8 pieces
    dict(s=513, m=36, e=5, k=2, dtype="f32", capacity=7, R=5),        # heavy drops, odd widths
    dict(s=700, m=16, e=12, k=3, dtype="f32", capacity=0, R=4),       # 3 experts per rank (not a power of 2)
    dict(s=1500, m=32, e=96, k=6, dtype="bf16", capacity=150, R=8),   # 12 experts per rank, drops
    dict(s=2049, m=64, e=64, k=6, dtype="bf16", capacity=200, R=8),
])
def test_edge_shapes(case):
    w = W.Workload("edge", seed=7, **case)
    full_parity(w, DEV)


@pytest.mark.parametrize("case", [
    dict(w=dict(s=1 << 17, m=16, e=256, k=4, dtype="bf16", capacity=0, R=8), priority="token"),
    dict(w=dict(s=70000, m=16, e=256, k=2, dtype="f32", capacity=300, R=4), priority="kmajor"),
    dict(w=dict(s=100000, m=8, e=128, k=8, dtype="bf16", capacity=5000, R=8), priority="token"),
], ids=["dropless-e256", "kmajor-capacity-e256", "capacity-e128"])
def test_many_subtile_layouts(case):
    """Batches long enough that each layout tile scans several 256-token
    sub-tiles (the look-back words are capped at 16384 = tiles x e), so the
    general sub-tile loop runs rather than the one- and two-sub-tile forms."""
    w = W.Workload("many-subtiles", seed=11, **case["w"])
    full_parity(w, DEV, priority=case["priority"])


def test_all_logits_equal_ties_and_drops():
    """Every token ties on every expert: all pick experts 0..k-1 (lower index
    wins), and capacity keeps only the first c tokens of each."""
    s, e, k, m, cap = 600, 8, 2, 64, 100
    logits = torch.zeros(s, e)
    idx, gate = B.moe_topk_gate(logits.to(DEV), k, 1)
    assert (bits(idx) == np.array([[0, 1]] * s)).all()
    assert (bits(gate) == 0.5).all()
    h = B.moe_dispatch_layout(idx, e, cap)
    L = oracle.layout(bits(idx), e, cap)
    check_layout(h, L, bits(idx))
    x = torch.randn(s, m, dtype=torch.float32)
    X = B.moe_dispatch(h, x.to(DEV))
    OX = oracle.dispatch(L["row"], x.numpy(), L["rows"])
    np.testing.assert_array_equal(bits(X), OX)
    og = np.full((s, k), 0.5, np.float32)
    out = B.moe_combine(h, to_dev(OX, DEV), to_dev(og, DEV))
    ref = oracle.combine(L["row"], og, OX)
    np.testing.assert_array_equal(bits(out)[cap:], 0)  # tokens past the capacity were fully dropped
    T.assert_close(bits(out), ref, T.combine_scale(L["row"], og, OX), "combine")


def test_empty_batch():
    for cap in (0, 3):
        idx = torch.empty(0, 2, dtype=torch.int32, device=DEV)
        h = B.moe_dispatch_layout(idx, 4, cap)
        assert h.rows == (4 * cap if cap else 0)
        assert bits(h.counts()).tolist() == [0, 0, 0, 0]
        assert bits(h.offsets()).tolist() == ([0, 3, 6, 9, 12] if cap else [0] * 5)
        x = torch.empty(0, 8, dtype=torch.bfloat16, device=DEV)
        X = B.moe_dispatch(h, x)
        if cap:
            assert X.shape == (12, 8) and (X == 0).all()
        out = B.moe_combine(h, X, torch.empty(0, 2, device=DEV))
        assert out.shape == (0, 8)
        assert h.status() == 0
        hs = B.moe_dispatch_layout_ex(idx, 4, cap, 2, send_slots=True)
        assert hs.rank_slot().shape == (0, 2) and bits(hs.rank_counts()).tolist() == [0, 0]
        xg = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
        Wg = torch.zeros(4, 256, 64, dtype=torch.bfloat16, device=DEV)
        Y = B.moe_dispatch_grouped_gemm(hs, xg, Wg)  # nothing to gather: no launch, no error
        assert Y.shape == (hs.rows, 256) and hs.status() == 0


@pytest.mark.parametrize("renorm", [0, 1])
@pytest.mark.parametrize("name", ["tiny-capacity", "mixtral-dropless", "fine-grained-skewed", "gshard-capacity",
                                  "diffusiongemma-replay"])
def test_gate_backward_parity(name, renorm):
    """Full token counts of each workload; the oracle's ids and gates and a
    seeded upstream gradient feed both sides."""
    w = W.WORKLOADS[name]
    logits = W.make_logits(w)
    oi, og = oracle.topk_gate(logits.numpy(), w.k, renorm)
    dgate = W.random_gates(w.s, w.k, seed=9).numpy() - 0.5
    dl = B.moe_topk_gate_bwd(logits.to(DEV) if not renorm else None, to_dev(oi, DEV), to_dev(og, DEV),
                             to_dev(dgate, DEV), w.e, renorm)
    ref = oracle.topk_gate_bwd(logits.numpy(), oi, og, dgate, w.e, renorm)
    got = bits(dl)
    T.assert_close(got, ref, T.gate_bwd_scale(oi, og, dgate, w.e, renorm, logits.numpy()), "dlogits")
    if renorm:
        sel = np.zeros_like(got, bool)
        np.put_along_axis(sel, oi.astype(np.int64), True, 1)
        assert np.all(got[~sel] == 0)


@pytest.mark.parametrize("renorm", [1, 0])
@pytest.mark.parametrize("name", list(REDUCED) + ["edge-k16", "edge-capacity-k6"])
def test_combine_gate_bwd_fused(name, renorm):
    """The combine backward with the gate backward fused in: dY and dgate
    against the oracle's combine backward, dlogits against the oracle's gate
    backward fed the kernel's own dgate (each op on identical inputs), and
    all three bit for bit equal to the two separate calls."""
    w = {"edge-k16": W.Workload("edge", s=301, m=64, e=64, k=16, dtype="bf16", capacity=0, R=0, seed=8),
         "edge-capacity-k6": W.Workload("edge", s=777, m=96, e=16, k=6, dtype="f32", capacity=200, R=0,
                                        seed=9)}.get(name) or REDUCED[name]
    inp = W.make_inputs(w)
    g = {k_: v.to(DEV) for k_, v in inp.items()}
    logits = inp["logits"].numpy()
    oi, og = oracle.topk_gate(logits, w.k, renorm)
    h = B.moe_dispatch_layout(to_dev(oi, DEV), w.e, w.capacity, w.R)
    L = oracle.layout(oi, w.e, w.capacity, w.R)
    gd = to_dev(og, DEV)
    dY, dgate, dl = B.moe_combine_gate_bwd(h, g["dout"], gd, g["y"], g["logits"], renorm)
    yb, db = bits(inp["y"]), bits(inp["dout"])
    row = L["row"]
    OdY, Odg = oracle.combine_bwd(row, og, db, yb)
    T.assert_close(bits(dY), OdY, np.abs(T.as_f64(OdY)), "dY")
    T.assert_close(bits(dgate), Odg, T.dot_scale(row, db, yb), "dgate")
    gdg = bits(dgate)
    Odl = oracle.topk_gate_bwd(logits, oi, og, gdg, w.e, renorm)
    T.assert_close(bits(dl), Odl, T.gate_bwd_scale(oi, og, gdg, w.e, renorm, logits), "dlogits")
    # the same bits as the two separate calls
    dY2, dgate2 = B.moe_combine_bwd(h, g["dout"], gd, g["y"])
    dl2 = B.moe_topk_gate_bwd(g["logits"] if not renorm else None, to_dev(oi, DEV), gd, dgate2, w.e, renorm)
    assert torch.equal(dY, dY2) and torch.equal(dgate, dgate2)
    assert torch.equal(dl.view(torch.int32), dl2.view(torch.int32))
    n = B.moe_launch_count("combine_gate_bwd")
    B.moe_combine_gate_bwd(h, g["dout"], gd, g["y"], g["logits"], renorm)
    assert B.moe_launch_count("combine_gate_bwd") == n + 1
    assert h.status() == 0


# ------------------------------------------------------------- full sizes --

@pytest.mark.parametrize("name", ["tiny-capacity", "mixtral-dropless", "fine-grained-skewed",
                                  "diffusiongemma-replay", "gshard-capacity"])
def test_full_size_workloads(name):
    """The exact workload shapes, in the launch configuration the benchmark
    times, compared in full: every index, count, gate, dispatched row (zero
    tails included), combined token, dY row, dgate and dx token against the
    oracle on the same inputs (DeepSpeed #8195, Testing: sparse against
    dense, element by element)."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device=DEV)
    logits = inp["logits"]
    idx, gate = B.moe_topk_gate(logits, w.k, w.renorm)
    oi, og = oracle.topk_gate(bits(logits), w.k, w.renorm)
    np.testing.assert_array_equal(bits(idx), oi)
    T.assert_gates_close(bits(gate), og)
    # from here on both sides take the oracle's routing and gates
    h = B.moe_dispatch_layout(to_dev(oi, DEV), w.e, w.capacity, w.R)
    L = oracle.layout(oi, w.e, w.capacity, w.R)
    check_layout(h, L, oi)
    gd = to_dev(og, DEV)
    row = L["row"]

    X = B.moe_dispatch(h, inp["x"])
    out = B.moe_combine(h, inp["y"], gd)
    dY, dgate = B.moe_combine_bwd(h, inp["dout"], gd, inp["y"])
    dx = B.moe_dispatch_bwd(h, inp["y"])  # the unit-weight combine of y
    torch.cuda.synchronize()
    assert h.status() == 0

    # dispatch: every row, bit-exact (capacity zero tails included)
    xb = bits(inp["x"])
    np.testing.assert_array_equal(bits(X), oracle.dispatch(row, xb, L["rows"]), err_msg="dispatch")
    del X, xb
    yb, db = bits(inp["y"]), bits(inp["dout"])
    T.assert_close(bits(out), oracle.combine(row, og, yb), lambda ts: T.combine_scale(row[ts], og[ts], yb), "combine")
    del out
    OdY, Odg = oracle.combine_bwd(row, og, db, yb)
    T.assert_close(bits(dY), OdY, lambda rs: np.abs(T.as_f64(OdY[rs])), "dY")
    T.assert_close(bits(dgate), Odg, lambda ts: T.dot_scale(row[ts], db[ts], yb), "dgate")
    del dY, OdY
    T.assert_close(bits(dx), oracle.dispatch_bwd(row, yb), lambda ts: T.combine_scale(row[ts], None, yb),
                   "dispatch_bwd")
    h.destroy()


# ----------------------------------------------------------- determinism --

def test_layout_rebuilds_are_bit_identical():
    w = W.WORKLOADS["fine-grained-skewed"]
    logits = W.make_logits(w, device=DEV)
    idx, _ = B.moe_topk_gate(logits, w.k)
    ref = None
    for _ in range(20):
        h = B.moe_dispatch_layout(idx, w.e, 0, w.R)
        got = [bits(getattr(h, n)()) for n in ("loc", "row", "counts", "offsets", "rank_counts")]
        if ref is None:
            ref = got
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)
        h.destroy()
    wc = W.WORKLOADS["gshard-capacity"]
    idx, _ = B.moe_topk_gate(W.make_logits(wc, device=DEV), wc.k)
    ref = None
    for _ in range(10):
        h = B.moe_dispatch_layout(idx, wc.e, wc.capacity)
        got = [bits(getattr(h, n)()) for n in ("loc", "row", "drop", "counts")]
        if ref is None:
            ref = got
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)


def test_replay_skips_layout_and_is_bit_identical():
    w = REDUCED["mixtral-dropless"]
    inp = W.make_inputs(w, device=DEV)
    idx, gate = B.moe_topk_gate(inp["logits"], w.k)
    h = B.moe_dispatch_layout(idx, w.e)
    X1 = B.moe_dispatch(h, inp["x"])
    o1 = B.moe_combine(h, inp["y"], gate)
    n_layout = B.moe_launch_count("layout")
    n_disp = B.moe_launch_count("dispatch")
    for _ in range(5):
        X2 = B.moe_dispatch(h, inp["x"])
        o2 = B.moe_combine(h, inp["y"], gate)
        assert torch.equal(X1, X2) and torch.equal(o1, o2)
    assert B.moe_launch_count("layout") == n_layout
    assert B.moe_launch_count("dispatch") == n_disp + 5


# --------------------------------------------------------- device errors --

def test_nonfinite_logits_are_flagged():
    logits = torch.randn(100, 16, device=DEV)
    logits[37, 3] = float("nan")
    logits[80, 0] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.moe_topk_gate(logits, 2, 1, device_status=status)
    assert int(status.item()) & B.MOE_DEV_NONFINITE
    status.zero_()
    B.moe_topk_gate(torch.randn(100, 16, device=DEV), 2, 1, device_status=status)
    assert int(status.item()) == 0


def test_bad_routes_are_flagged_not_followed():
    idx = torch.tensor([[0, 1], [2, 2], [5, 1], [-1, 3], [3, 0]], dtype=torch.int32, device=DEV)
    h = B.moe_dispatch_layout(idx, 4)
    assert h.status() & B.MOE_DEV_BAD_ROUTE
    row = bits(h.row())
    assert row[1, 1] == -1 and row[2, 0] == -1 and row[3, 0] == -1  # repeat, out of range, negative
    assert row[1, 0] >= 0 and row[0, 0] >= 0
    kept = row[row >= 0]
    assert len(np.unique(kept)) == len(kept)
    X = B.moe_dispatch(h, torch.ones(5, 8, device=DEV))  # must not fault
    torch.cuda.synchronize()


def test_layout_wait_times_out_without_hanging():
    """A tile that never publishes: later tiles' bounded waits run out, the
    handle reports MOE_DEV_TIMEOUT, and the context stays usable."""
    s, e, k = 256 * 6, 8, 2
    idx = W.random_routes(s, e, k, device=DEV, seed=1)
    B.moe_debug_hold_layout_tile(2, timeout_ms=200)
    h = B.moe_dispatch_layout(idx, e)
    assert h.status() & B.MOE_DEV_TIMEOUT
    h.destroy()
    h = B.moe_dispatch_layout(idx, e)  # the hook disarmed itself
    assert h.status() == 0
    check_layout(h, oracle.layout(bits(idx), e), bits(idx))


# -------------------------------------------------------------- host API --

def test_host_validation_on_device():
    x = torch.randn(4, 8, device=DEV)
    idx = torch.tensor([[0, 1]] * 4, dtype=torch.int32, device=DEV)
    h = B.moe_dispatch_layout(idx, 2)
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch(h, x.half())
    assert ei.value.name == "MOE_ERR_DTYPE"
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch(h, torch.randn(5, 8, device=DEV))
    assert ei.value.name == "MOE_ERR_HANDLE_MISMATCH"
    with pytest.raises(B.MoEError) as ei:
        B.moe_combine(h, torch.randn(7, 8, device=DEV), torch.ones(4, 2, device=DEV))
    assert ei.value.name == "MOE_ERR_HANDLE_MISMATCH"
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch(h, torch.randn(4, 8))  # host memory
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch(h, torch.randn(4, 6, device=DEV))  # 24-byte rows
    assert ei.value.name == "MOE_ERR_INVALID_ARG"
    raw = h.raw
    h.destroy()
    import ctypes

    rc = B.lib().moe_dispatch(raw, 4, 8, 8, B.MOE_F32, ctypes.c_void_p(x.data_ptr()), None, None)
    assert B.STATUS[rc] == "MOE_ERR_HANDLE_MISMATCH"
