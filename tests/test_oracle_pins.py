"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle (``oracle/``) against a value fixed by the pages
or by mathematics: a hand-worked example (``tests/golden``), brute-force
enumeration, a closed form (the cumulative-sum formula for locations), a
library routine (NumPy stable sort, SciPy softmax, torch's bf16 rounding,
a dense one-hot einsum in float64), conservation invariants, adjoint
identities and finite differences.  Each is chosen so that a plausible slip
in the oracle (off-by-one location, k-major instead of token-order priority,
a missing gate, a transposed operand, a wrong sign) fails at least one.

Sources: DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption,
speed up native and Tutel paths" (changes 1 and 3, Testing); DeepSpeed #8213
"Add an opt-in DeepEP transport for the AutoEP expert all-to-all"
(description; review thread on weighted combine and router gradients).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from combine_moe_topk_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0**-126)))
    return 2.0 ** (e - 7)


# ------------------------------------------------------------------ golden --

def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_s4_e3_k2.json")))
    logits = np.array(g["logits"], np.float32)
    k = g["k"]
    idx, gate = oracle.topk_gate(logits, k, renorm=1)
    assert idx.tolist() == g["idx"]
    np.testing.assert_allclose(gate, np.array(g["gate_renorm"]), rtol=1e-7)
    idx0, gate0 = oracle.topk_gate(logits, k, renorm=0)
    assert idx0.tolist() == g["idx"]
    np.testing.assert_allclose(gate0, np.array(g["gate_full_softmax"]), rtol=1e-7)

    cap = g["capacity"]
    L = oracle.layout(idx, e=3, capacity=cap["c"], R=3)
    assert L["loc"].tolist() == g["loc"]
    assert L["raw_counts"].tolist() == g["raw_counts"]
    assert L["drop"].tolist() == cap["drop"]
    assert L["counts"].tolist() == cap["counts"]
    assert L["offsets"].tolist() == cap["offsets"]
    assert L["row"].tolist() == cap["row"]
    assert L["token_in_rank"].tolist() == cap["token_in_rank_R3"]
    assert L["rank_counts"].tolist() == cap["rank_counts_R3"]
    assert L["rank_slot"].tolist() == cap["rank_slot_R3"]

    dl = g["dropless"]
    L = oracle.layout(idx, e=3, capacity=0, R=3)
    assert L["loc"].tolist() == g["loc"]
    assert L["drop"].sum() == 0
    assert L["counts"].tolist() == dl["counts"]
    assert L["offsets"].tolist() == dl["offsets"]
    assert L["row"].tolist() == dl["row"]
    assert L["token_in_rank"].tolist() == dl["token_in_rank_R3"]
    assert L["rank_counts"].tolist() == dl["rank_counts_R3"]
    assert L["rank_slot"].tolist() == dl["rank_slot_R3"]


# -------------------------------------------------------------------- bf16 --

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    vals = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895313892515355e38, 3.4e38, -3.4e38,
            1e-40, -1e-40, 1.17549435e-38, 2.0**-133]
    # exact ties: the low 16 bits are 0x8000, with the kept lsb even and odd
    for hi in (0x3F80, 0x3F81, 0xBF80, 0xBF81, 0x7F7F, 0x0001, 0x0080):
        vals.append(np.array([(hi << 16) | 0x8000], np.uint32).view(np.float32)[0])
        vals.append(np.array([(hi << 16) | 0x7FFF], np.uint32).view(np.float32)[0])
        vals.append(np.array([(hi << 16) | 0x8001], np.uint32).view(np.float32)[0])
    vals += list(rng.standard_normal(3000).astype(np.float32))
    vals += list((rng.standard_normal(2000) * 1e30).astype(np.float32))
    vals += list(rng.integers(0, 2**32, 3000, dtype=np.uint64).astype(np.uint32).view(np.float32))
    f = np.array(vals, np.float32)
    ref = bf16_bits(torch.from_numpy(f).to(torch.bfloat16))
    got = np.array([oracle.f32_to_bf16(float(v)) for v in f], np.uint16)
    nan = np.isnan(f)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(bits_to_f64(got[nan])))
    # widening is exact
    for b in rng.integers(0, 2**16, 2000):
        v = oracle.bf16_to_f32(int(b))
        w = float(torch.tensor([int(b)], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float())
        assert (math.isnan(v) and math.isnan(w)) or v == w


# -------------------------------------------------------------------- gate --

@pytest.mark.parametrize("s,e,k", [(64, 8, 2), (50, 128, 8), (33, 64, 6), (20, 5, 5), (40, 256, 16), (7, 1, 1)])
def test_topk_matches_stable_sort(s, e, k):
    rng = np.random.default_rng(s * 1000 + e)
    logits = rng.standard_normal((s, e)).astype(np.float32)
    # plant ties, including +0.0 against -0.0
    logits[0, : min(e, 4)] = 0.5
    if e >= 3:
        logits[1, 0], logits[1, 2] = -0.0, 0.0
        logits[1, 1] = -1.0
    logits[2 % s] = np.round(logits[2 % s])
    idx, gate = oracle.topk_gate(logits, k)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(idx, ref)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(7)
    for _ in range(200):
        e = int(rng.integers(1, 9))
        k = int(rng.integers(1, e + 1))
        l = rng.integers(-2, 3, size=e).astype(np.float32)  # many ties
        idx, _ = oracle.topk_gate(l[None], k)
        # enumerate: best k under (value desc, index asc)
        order = sorted(range(e), key=lambda j: (-float(l[j]), j))
        assert idx[0].tolist() == order[:k]


@pytest.mark.parametrize("renorm", [0, 1])
def test_gates_match_scipy_softmax(renorm):
    rng = np.random.default_rng(11 + renorm)
    s, e, k = 300, 64, 6
    logits = (rng.standard_normal((s, e)) * 3).astype(np.float32)
    idx, gate = oracle.topk_gate(logits, k, renorm=renorm)
    l64 = logits.astype(np.float64)
    if renorm:
        ref = scipy.special.softmax(np.take_along_axis(l64, idx, 1), axis=1)
    else:
        ref = np.take_along_axis(scipy.special.softmax(l64, axis=1), idx, 1)
    # the oracle rounds once from double: at most one float ulp away
    np.testing.assert_array_less(np.abs(gate - ref.astype(np.float32)), np.spacing(np.abs(ref.astype(np.float32))) * 1.01)
    if renorm:
        np.testing.assert_allclose(gate.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(gate, axis=1) <= 0), "gates follow the descending logits"


def test_gates_special_cases():
    # all logits equal: ties to the lower index; gates 1/k (renorm) or 1/e
    l = np.full((3, 8), 0.25, np.float32)
    idx, g = oracle.topk_gate(l, 3, renorm=1)
    assert idx.tolist() == [[0, 1, 2]] * 3
    np.testing.assert_allclose(g, 1 / 3, rtol=1e-7)
    _, g0 = oracle.topk_gate(l, 3, renorm=0)
    np.testing.assert_allclose(g0, 1 / 8, rtol=1e-7)
    # k = e without renormalisation is the full softmax, sorted
    rng = np.random.default_rng(3)
    l = rng.standard_normal((5, 7)).astype(np.float32)
    idx, g = oracle.topk_gate(l, 7, renorm=0)
    ref = scipy.special.softmax(l.astype(np.float64), axis=1)
    np.testing.assert_allclose(g, np.take_along_axis(ref, idx, 1), rtol=2e-7)
    # k = 1 with renorm gives weight exactly one
    _, g1 = oracle.topk_gate(l, 1, renorm=1)
    assert np.all(g1 == 1.0)


def test_gate_rejects_nonfinite():
    l = np.zeros((2, 4), np.float32)
    l[1, 2] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.topk_gate(l, 2)
    l[1, 2] = np.inf
    with pytest.raises(oracle.OracleError):
        oracle.topk_gate(l, 2)


# ------------------------------------------------------------------ layout --

def brute_layout(idx, e, capacity):
    s, k = idx.shape
    loc = np.zeros_like(idx)
    for t in range(s):
        for j in range(k):
            x = idx[t, j]
            loc[t, j] = sum(1 for t2 in range(t) for j2 in range(k) if idx[t2, j2] == x)
    return loc


def cumsum_locations(idx, e):
    """The pages' formula: location = cumulative sum (over tokens) of the
    one-hot expert mask, minus one, read at each route."""
    s, k = idx.shape
    mask = np.zeros((s, e), np.int64)
    np.put_along_axis(mask, idx.astype(np.int64), 1, axis=1)
    cum = np.cumsum(mask, axis=0) - 1
    return np.take_along_axis(cum, idx.astype(np.int64), 1).astype(np.int32)


@pytest.mark.parametrize("s,e,k,cap", [(40, 8, 2, 0), (40, 8, 2, 6), (30, 16, 4, 5), (25, 6, 6, 3), (1, 4, 2, 1), (0, 4, 2, 0)])
def test_layout_brute_force(s, e, k, cap):
    idx = W.random_routes(s, e, k, seed=s + e).numpy() if s else np.zeros((0, k), np.int32)
    L = oracle.layout(idx, e, cap)
    np.testing.assert_array_equal(L["loc"], brute_layout(idx, e, cap))
    if s:
        np.testing.assert_array_equal(L["loc"], cumsum_locations(idx, e))


def check_invariants(idx, e, cap, L):
    s, k = idx.shape
    loc, row, drop = L["loc"], L["row"], L["drop"].astype(bool)
    raw, counts, off = L["raw_counts"], L["counts"], L["offsets"]
    rows = e * cap if cap else s * k
    assert raw.sum() == s * k
    np.testing.assert_array_equal(raw, np.bincount(idx.ravel(), minlength=e))
    assert counts.sum() == s * k - drop.sum()
    kept = row[~drop]
    assert len(np.unique(kept)) == len(kept), "every kept route owns a unique row"
    assert np.all((kept >= 0) & (kept < rows))
    assert np.all(row[drop] == -1)
    if cap:
        assert np.all(counts <= cap)
        np.testing.assert_array_equal(drop, loc >= cap)
        np.testing.assert_array_equal(counts, np.minimum(raw, cap))
    else:
        assert not drop.any()
        assert off[0] == 0 and off[-1] == rows
        np.testing.assert_array_equal(np.diff(off), counts)
    # slots fill in token order within each expert
    for x in range(e):
        t_of = np.nonzero((idx == x).any(1))[0]
        locs = loc[idx == x]  # row-major order = token order
        np.testing.assert_array_equal(locs, np.arange(len(t_of)))
        if not cap:
            np.testing.assert_array_equal(row[idx == x], off[x] + np.arange(len(t_of)))


@pytest.mark.parametrize("name", ["tiny-capacity", "mixtral-dropless", "fine-grained-skewed", "gshard-capacity"])
def test_layout_invariants_on_workload_routing(name):
    w = W.WORKLOADS[name]
    w = w.replace(s=min(w.s, 4096))
    cap = w.capacity if w.capacity == 0 else max(1, (w.capacity * w.s) // W.WORKLOADS[name].s)
    logits = W.make_logits(w).numpy()
    idx, _ = oracle.topk_gate(logits, w.k)
    L = oracle.layout(idx, w.e, cap, R=w.R)
    check_invariants(idx, w.e, cap, L)
    np.testing.assert_array_equal(L["loc"], cumsum_locations(idx, w.e))


@pytest.mark.parametrize("cap,R", [(0, 4), (3, 4), (0, 1), (2, 8), (0, 8)])
def test_dedup_brute_force(cap, R):
    s, e, k = 60, 16, 4
    idx = W.random_routes(s, e, k, seed=5).numpy()
    L = oracle.layout(idx, e, cap, R=R)
    per = e // R
    tir = np.zeros((s, R), np.uint8)
    for t in range(s):
        for j in range(k):
            if not L["drop"][t, j]:
                tir[t, idx[t, j] // per] = 1
    np.testing.assert_array_equal(L["token_in_rank"], tir)
    np.testing.assert_array_equal(L["rank_counts"], tir.sum(0))
    u = int((~L["drop"].astype(bool)).any(1).sum())
    assert u <= L["rank_counts"].sum() <= s * min(k, R)
    for r in range(R):
        assert L["rank_counts"][r] <= L["counts"][r * per:(r + 1) * per].sum()


def test_layout_rejects_bad_routes():
    with pytest.raises(oracle.OracleError):
        oracle.layout(np.array([[0, 4]], np.int32), e=4)
    with pytest.raises(oracle.OracleError):
        oracle.layout(np.array([[1, 1]], np.int32), e=4)
    with pytest.raises(oracle.OracleError):
        oracle.layout(np.array([[-1, 1]], np.int32), e=4)


# ------------------------------------------------------- dispatch / combine --

def dense_masks(idx, L, e, cap, gate):
    """One-hot [s, rows] route mask and its gate-weighted twin, float64.
    With capacity this is the [s, e, c] mask of the dense einsum path,
    flattened over (e, c)."""
    s, k = idx.shape
    rows = e * cap if cap else s * k
    mask = np.zeros((s, rows))
    gm = np.zeros((s, rows))
    for t in range(s):
        for j in range(k):
            if not L["drop"][t, j]:
                x, l = int(idx[t, j]), int(L["loc"][t, j])
                r = x * cap + l if cap else int(L["offsets"][x]) + l
                mask[t, r] = 1.0
                gm[t, r] = float(gate[t, j])
    return mask, gm


def to64(a):
    return bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def draw(shape, dtype, rng):
    v = rng.standard_normal(shape).astype(np.float32)
    return bf16_bits(torch.from_numpy(v).to(torch.bfloat16)) if dtype == "bf16" else v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("s,e,k,cap", [(48, 8, 2, 10), (48, 8, 2, 0), (40, 16, 4, 0), (37, 6, 3, 4)])
def test_dispatch_combine_match_dense_einsum(dtype, s, e, k, cap):
    rng = np.random.default_rng(s + 100 * e + cap)
    m = 24
    idx = W.random_routes(s, e, k, seed=s + e).numpy()
    gate = (rng.random((s, k)) + 0.05).astype(np.float32)
    L = oracle.layout(idx, e, cap)
    rows = L["rows"]
    x = draw((s, m), dtype, rng)
    y = draw((rows, m), dtype, rng)
    mask, gm = dense_masks(idx, L, e, cap, gate)
    if cap:
        # the [s, e, c] einsum of the dense path, written with torch
        mask3 = torch.from_numpy(mask.reshape(s, e, cap))
        Xd = torch.einsum("sec,sm->ecm", mask3, torch.from_numpy(to64(x))).reshape(rows, m).numpy()
        gm3 = torch.from_numpy(gm.reshape(s, e, cap))
        outd = torch.einsum("sec,ecm->sm", gm3, torch.from_numpy(to64(y)).reshape(e, cap, m)).numpy()
    else:
        Xd = mask.T @ to64(x)
        outd = gm @ to64(y)

    X = oracle.dispatch(L["row"], x, rows)
    np.testing.assert_array_equal(to64(X), Xd)  # a copy: exact

    out = oracle.combine(L["row"], gate, y)
    scale = np.abs(gm) @ np.abs(to64(y))
    err = np.abs(to64(out) - outd)
    if dtype == "f32":
        assert np.all(err <= 1e-6 * scale + 1e-30)
    else:
        assert np.all(err <= bf16_ulp(outd) + 1e-30)
    # the weights are applied: the unweighted sum is different
    unweighted = mask @ to64(y)
    assert np.abs(unweighted - outd).max() > 1e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cap", [0, 5])
def test_backward_adjoints_and_finite_difference(dtype, cap):
    rng = np.random.default_rng(21 + cap)
    s, e, k, m = 40, 8, 3, 16
    idx = W.random_routes(s, e, k, seed=9).numpy()
    gate = (rng.random((s, k)) + 0.05).astype(np.float32)
    L = oracle.layout(idx, e, cap)
    rows = L["rows"]
    x = draw((s, m), dtype, rng)
    y = draw((rows, m), dtype, rng)
    dout = draw((s, m), dtype, rng)
    dXin = draw((rows, m), dtype, rng)
    mask, gm = dense_masks(idx, L, e, cap, gate)
    tol = 1e-6 if dtype == "f32" else 1e-2

    # <dispatch(x), dX> = <x, dispatch_bwd(dX)>
    X = to64(oracle.dispatch(L["row"], x, rows))
    dx = to64(oracle.dispatch_bwd(L["row"], dXin))
    lhs, rhs = np.sum(X * to64(dXin)), np.sum(to64(x) * dx)
    assert abs(lhs - rhs) <= tol * np.sum(np.abs(mask.T @ np.abs(to64(x))) * np.abs(to64(dXin)))
    # dispatch_bwd is the unit-weight combine: the transpose of the dispatch mask
    ref = mask @ to64(dXin)
    if dtype == "f32":
        assert np.all(np.abs(dx - ref) <= 1e-6 * (mask @ np.abs(to64(dXin))) + 1e-30)
    else:
        assert np.all(np.abs(dx - ref) <= bf16_ulp(ref) + 1e-30)

    # <combine(y), dout> = <y, dY>
    dY, dgate = oracle.combine_bwd(L["row"], gate, dout, y)
    out = gm @ to64(y)
    lhs = np.sum(out * to64(dout))
    rhs = np.sum(to64(y) * to64(dY))
    assert abs(lhs - rhs) <= tol * np.sum(np.abs(gm) @ np.abs(to64(y)) * np.abs(to64(dout)))
    # dY is the gate-scaled scatter of dout; untouched rows are zero
    dYd = gm.T @ to64(dout)
    err = np.abs(to64(dY) - dYd)
    assert np.all(err <= (1e-6 * np.abs(dYd) if dtype == "f32" else bf16_ulp(dYd)) + 1e-30)
    assert np.all(to64(dY)[mask.sum(0) == 0] == 0)

    # dgate is the derivative of <combine(y, gate), dout> in each gate (central difference, float64)
    y64, d64 = to64(y), to64(dout)

    def loss(g):
        _, gmm = dense_masks(idx, L, e, cap, g)
        return np.sum((gmm @ y64) * d64)

    h = 1e-3
    for t, j in [(0, 0), (3, 1), (s - 1, k - 1), (17, 2)]:
        gp, gn = gate.astype(np.float64).copy(), gate.astype(np.float64).copy()
        gp[t, j] += h
        gn[t, j] -= h
        fd = (loss(gp) - loss(gn)) / (2 * h)
        scale = np.sum(np.abs(d64[t])) * np.abs(y64).max() + 1e-30
        if L["drop"][t, j]:
            assert dgate[t, j] == 0.0 and abs(fd) < 1e-9
        else:
            assert abs(dgate[t, j] - fd) <= 1e-6 * scale


def test_identity_expert_returns_input():
    """Dropless, gates renormalised to one, y = dispatch(x): combine gives x back."""
    rng = np.random.default_rng(4)
    s, e, k, m = 64, 16, 4, 32
    logits = rng.standard_normal((s, e)).astype(np.float32)
    idx, gate = oracle.topk_gate(logits, k, renorm=1)
    L = oracle.layout(idx, e, 0)
    for dtype in ("f32", "bf16"):
        x = draw((s, m), dtype, rng)
        X = oracle.dispatch(L["row"], x, L["rows"])
        out = oracle.combine(L["row"], gate, X)
        if dtype == "f32":
            np.testing.assert_allclose(out, x, rtol=1e-6, atol=1e-30)
        else:
            np.testing.assert_array_equal(out, x)


def test_tiny_workload_with_the_affine_expert():
    """The tiny capacity workload as specified (seed 0, s=256, m=128, e=8,
    k=2, fp32, capacity 80, token order with drops) with its expert
    y = 2*X + 1 on the dispatched buffer: the combine must give
    (sum of the token's kept gates) * (2 x + 1) -- exactly 2 x + 1 (to fp32
    rounding) where both routes are kept, zero where both are dropped.  A
    dropped gate still added, a kept one skipped, or the wrong row read
    fails it."""
    w = W.WORKLOADS["tiny-capacity"]
    inp = W.make_inputs(w, with_grad=False)
    logits, x = inp["logits"].numpy(), inp["x"].numpy()
    idx, gate = oracle.topk_gate(logits, w.k, w.renorm)
    L = oracle.layout(idx, w.e, w.capacity)
    assert L["rows"] == 640 and L["drop"].any() and not L["drop"].all()
    X = oracle.dispatch(L["row"], x, L["rows"])
    y = np.float32(2.0) * X + np.float32(1.0)
    out = oracle.combine(L["row"], gate, y).astype(np.float64)
    kept = L["row"] >= 0
    kg = np.where(kept, gate.astype(np.float64), 0.0).sum(axis=1, keepdims=True)
    affine = 2.0 * x.astype(np.float64) + 1.0
    assert np.all(np.abs(out - kg * affine) <= 4 * 2.0**-24 * np.abs(kg) * np.abs(affine) + 1e-30)
    both = kept.all(axis=1)
    assert both.any() and np.all(np.abs(out[both] - affine[both]) <= 1e-6 * np.abs(affine[both]))
    assert np.all(out[~kept.any(axis=1)] == 0)


def test_fully_dropped_token_gives_zero():
    idx = np.array([[0, 1], [0, 1], [0, 1]], np.int32)
    L = oracle.layout(idx, e=2, capacity=1)
    assert L["drop"].tolist() == [[0, 0], [1, 1], [1, 1]]
    y = np.arange(2 * 1 * 4, dtype=np.float32).reshape(2, 4) + 1
    gate = np.full((3, 2), 0.5, np.float32)
    out = oracle.combine(L["row"], gate, y)
    assert np.all(out[1:] == 0) and np.all(out[0] == 0.5 * (y[0] + y[1]))
    dY, dg = oracle.combine_bwd(L["row"], gate, np.ones((3, 4), np.float32), y)
    assert np.all(dg[1:] == 0)


def test_combine_accumulates_in_fp32_k_order():
    """Three routes whose fp32 sum depends on the order: the definition
    (fmaf in route order, starting from +0) fixes the bits."""
    y = np.array([[1.0], [2.0**-24], [2.0**-24]], np.float32)
    row = np.array([[0, 1, 2]], np.int32)
    g = np.ones((1, 3), np.float32)
    out = oracle.combine(row, g, y)
    # 1 + 2^-24 rounds to 1 (tie to even), twice: order 0,1,2 gives exactly 1
    assert out[0, 0] == np.float32(1.0)
    out2 = oracle.combine(np.array([[1, 2, 0]], np.int32), g, y)
    assert out2[0, 0] == np.float32(1.0 + 2.0**-23)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(8)
    s, e, k, m = 200, 16, 4, 64
    logits = rng.standard_normal((s, e)).astype(np.float32)
    y = rng.standard_normal((s * k, m)).astype(np.float32)
    outs = []
    for n in (1, 4):
        oracle.set_threads(n)
        idx, gate = oracle.topk_gate(logits, k)
        L = oracle.layout(idx, e)
        outs.append((idx, gate, oracle.combine(L["row"], gate, y)))
    oracle.set_threads(1)
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------ gate backward --

def gate_forward_f64(logits, idx, renorm):
    """The gates as a function of the logits with the selection held fixed,
    written with SciPy's softmax (float64)."""
    l = logits.astype(np.float64)
    if renorm:
        return scipy.special.softmax(np.take_along_axis(l, idx.astype(np.int64), 1), axis=1)
    return np.take_along_axis(scipy.special.softmax(l, axis=1), idx.astype(np.int64), 1)


@pytest.mark.parametrize("renorm", [0, 1])
def test_gate_backward_matches_central_differences(renorm):
    rng = np.random.default_rng(40 + renorm)
    s, e, k = 12, 16, 4
    logits = rng.standard_normal((s, e)).astype(np.float32)
    idx, gate = oracle.topk_gate(logits, k, renorm=renorm)
    dgate = rng.standard_normal((s, k)).astype(np.float32)
    dl = oracle.topk_gate_bwd(logits, idx, gate, dgate, e, renorm)
    h = 1e-5
    for t in range(s):
        for i in range(e):
            lp, ln = logits.astype(np.float64).copy(), logits.astype(np.float64).copy()
            lp[t, i] += h
            ln[t, i] -= h
            fd = (np.sum(gate_forward_f64(lp, idx, renorm)[t] * dgate[t]) -
                  np.sum(gate_forward_f64(ln, idx, renorm)[t] * dgate[t])) / (2 * h)
            assert abs(dl[t, i] - fd) <= 1e-6 + 1e-5 * abs(fd), (t, i, dl[t, i], fd)
    if renorm:
        sel = np.zeros((s, e), bool)
        np.put_along_axis(sel, idx.astype(np.int64), True, 1)
        assert np.all(dl[~sel] == 0), "experts outside the top-k get no gradient"
    # softmax gradients sum to zero over the logits they depend on
    np.testing.assert_allclose(dl.astype(np.float64).sum(1), 0, atol=1e-6)


def test_gate_backward_special_cases():
    # k = 1 with renorm: the gate is constant 1, so no gradient at all
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((5, 8)).astype(np.float32)
    idx, gate = oracle.topk_gate(logits, 1, renorm=1)
    dl = oracle.topk_gate_bwd(logits, idx, gate, rng.standard_normal((5, 1)).astype(np.float32), 8, 1)
    assert np.all(dl == 0)
    # uniform upstream gradient with renorm: sum of gates is 1, so again zero
    idx, gate = oracle.topk_gate(logits, 3, renorm=1)
    dl = oracle.topk_gate_bwd(logits, idx, gate, np.full((5, 3), 2.5, np.float32), 8, 1)
    np.testing.assert_allclose(dl, 0, atol=1e-7)
    # k = e without renorm is the full softmax Jacobian-vector product: p*(v - <p, v>)
    idx, gate = oracle.topk_gate(logits, 8, renorm=0)
    v = rng.standard_normal((5, 8)).astype(np.float32)
    dl = oracle.topk_gate_bwd(logits, idx, gate, v, 8, 0)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    vf = np.zeros((5, 8))
    np.put_along_axis(vf, idx.astype(np.int64), v.astype(np.float64), 1)
    ref = p * (vf - np.sum(p * vf, axis=1, keepdims=True))
    np.testing.assert_allclose(dl, ref, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------- layout variants --

def brute_kmajor_loc(idx):
    s, k = idx.shape
    loc = np.zeros_like(idx)
    for t in range(s):
        for j in range(k):
            x = idx[t, j]
            loc[t, j] = sum(1 for t2 in range(s) for j2 in range(k)
                            if idx[t2, j2] == x and (j2 < j or (j2 == j and t2 < t)))
    return loc


@pytest.mark.parametrize("cap", [0, 4])
def test_kmajor_priority_brute_force(cap):
    idx = W.random_routes(30, 6, 3, seed=12).numpy()
    L = oracle.layout(idx, 6, cap, priority=1)
    np.testing.assert_array_equal(L["loc"], brute_kmajor_loc(idx))
    # closed form: the token-order formula applied to the slot-major route list
    flat = np.ascontiguousarray(idx.T).reshape(-1, 1)
    np.testing.assert_array_equal(L["loc"].T.reshape(-1, 1), cumsum_locations(flat, 6))
    check_invariants_kmajor(idx, 6, cap, L)


def check_invariants_kmajor(idx, e, cap, L):
    s, k = idx.shape
    drop = L["drop"].astype(bool)
    assert L["raw_counts"].sum() == s * k
    assert L["counts"].sum() == s * k - drop.sum()
    kept = L["row"][~drop]
    assert len(np.unique(kept)) == len(kept)
    if cap:
        # first choices are never dropped while a later choice to the same expert is kept
        for x in range(e):
            first_dropped = drop[:, 0] & (idx[:, 0] == x)
            later_kept = (~drop[:, 1:]) & (idx[:, 1:] == x)
            assert not (first_dropped.any() and later_kept.any())


def test_kmajor_differs_from_token_order_and_matches_hand_example():
    # the hand-worked example, k-major: expert 0 gets t1 (1st choice), t2 (1st),
    # then t3 (2nd); expert 1 gets t0 (1st), t3 (1st), then t1 (2nd)
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_s4_e3_k2.json")))
    idx = np.array(g["idx"], np.int32)
    L = oracle.layout(idx, 3, 0, priority=1)
    assert L["loc"].tolist() == [[0, 0], [0, 2], [1, 1], [1, 2]]
    assert L["loc"].tolist() != g["loc"]


@pytest.mark.parametrize("P", [1, 4, 128])
def test_pad_multiple_offsets(P):
    idx = W.random_routes(200, 8, 2, seed=3).numpy()
    L = oracle.layout(idx, 8, 0, pad_multiple=P)
    counts = L["counts"]
    seg = np.diff(L["offsets"])
    assert np.all(seg % P == 0) and np.all(seg >= counts) and np.all(seg - counts < P)
    assert L["offsets"][0] == 0 and L["offsets"][-1] <= L["rows"] == 200 * 2 + 8 * (P - 1)
    base = oracle.layout(idx, 8, 0)
    np.testing.assert_array_equal(L["loc"], base["loc"])
    np.testing.assert_array_equal(L["row"], L["offsets"][idx] + L["loc"])
    with pytest.raises(oracle.OracleError):
        oracle.layout(idx, 8, capacity=10, pad_multiple=4)


# ------------------------------------------------ grouped GEMM consumer --
# DeepSpeed #8213 description: the arrivals are grouped by expert for a
# grouped GEMM bounded by offsets.  The oracle multiplies each owned row by
# its own expert's weight, transposed (W [e, N, K]).

GEMM_CAP = 40


def _gemm_layout():
    idx = W.random_routes(60, 3, 2, seed=11).numpy()
    L = oracle.layout(idx, 3, capacity=GEMM_CAP)
    # both cases present: an expert that drops, and one with a tail no route owns
    assert (L["raw_counts"] > GEMM_CAP).any() and (L["counts"] < GEMM_CAP).any()
    return L


def test_grouped_gemm_identity_weights_return_owned_rows():
    L = _gemm_layout()
    rng = np.random.default_rng(0)
    X = rng.standard_normal((L["rows"], 6)).astype(np.float32)
    Y = oracle.grouped_gemm(X, np.stack([np.eye(6, dtype=np.float32)] * 3), L["offsets"], L["counts"])
    for x in range(3):
        o, n = int(L["offsets"][x]), int(L["counts"][x])
        np.testing.assert_array_equal(Y[o:o + n], X[o:o + n].astype(np.float64))
        assert np.isnan(Y[o + n:o + GEMM_CAP]).all()  # rows past counts[x] are nobody's


def test_grouped_gemm_uses_each_segments_own_weight_untransposed():
    # W[x] = (x + 1) * P with P a non-symmetric permutation: Y[r, i] must be
    # (x + 1) * X[r, p(i)].  Another expert's weight scales wrongly; P^T
    # (a transposed operand) permutes the other way.
    L = _gemm_layout()
    K = 5
    p = np.array([1, 2, 3, 4, 0])
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), p] = 1.0
    assert not np.array_equal(P, P.T)
    rng = np.random.default_rng(1)
    X = rng.standard_normal((L["rows"], K)).astype(np.float32)
    Y = oracle.grouped_gemm(X, np.stack([(x + 1) * P for x in range(3)]), L["offsets"], L["counts"])
    for x in range(3):
        o, n = int(L["offsets"][x]), int(L["counts"][x])
        np.testing.assert_array_equal(Y[o:o + n], (x + 1) * X[o:o + n][:, p].astype(np.float64))


def test_grouped_gemm_brute_force_and_bf16_decoding():
    idx = np.array([[0, 2], [1, 2], [2, 0], [2, 1]], np.int32)
    L = oracle.layout(idx, 3, 0)
    Xb = torch.randn(L["rows"], 4, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    Wb = torch.randn(3, 2, 4, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    Xbits = Xb.view(torch.int16).numpy().view(np.uint16)
    Wbits = Wb.view(torch.int16).numpy().view(np.uint16)
    Y = oracle.grouped_gemm(Xbits, Wbits, L["offsets"], L["counts"])
    Xv, Wv = Xb.double().tolist(), Wb.double().tolist()
    for x in range(3):
        for r in range(int(L["offsets"][x]), int(L["offsets"][x + 1])):
            for n in range(2):
                want = math.fsum(Xv[r][kk] * Wv[x][n][kk] for kk in range(4))
                assert abs(Y[r, n] - want) <= 1e-12 * (1 + abs(want))
    # the same values as float32 give the same result
    np.testing.assert_array_equal(Y, oracle.grouped_gemm(Xb.float().numpy(), Wb.float().numpy(),
                                                         L["offsets"], L["counts"]))


# ------------------------------------------------ per-rank send slots --
# DeepSpeed #8213 description: a token is sent to a destination rank once;
# its place in that rank's send buffer is its token-order rank among the
# tokens that go there.

@pytest.mark.parametrize("cap", [0, 30])
def test_rank_slots_brute_force_and_invariants(cap):
    idx = W.random_routes(300, 16, 4, seed=21).numpy()
    R = 4
    L = oracle.layout(idx, 16, cap, R)
    tir, slot = L["token_in_rank"], L["rank_slot"]
    s = idx.shape[0]
    for r in range(R):
        for t in range(0, s, 7):
            want = sum(int(tir[t2, r]) for t2 in range(t)) if tir[t, r] else -1
            assert slot[t, r] == want
        used = np.sort(slot[:, r][slot[:, r] >= 0])
        np.testing.assert_array_equal(used, np.arange(L["rank_counts"][r]))  # a permutation of 0..n-1
    assert ((slot >= 0) == tir.astype(bool)).all()
    if cap:
        assert L["drop"].any()  # drops change which tokens send where


def test_rank_slots_closed_form():
    # slot = inclusive cumulative sum of the column - 1, where the token sends
    tir = (np.random.default_rng(5).random((500, 8)) < 0.3).astype(np.uint8)
    slot = oracle.rank_slots(tir)
    want = np.where(tir == 1, np.cumsum(tir.astype(np.int64), axis=0) - 1, -1)
    np.testing.assert_array_equal(slot, want)
