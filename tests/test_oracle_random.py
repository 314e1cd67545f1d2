"""Randomised pins of the oracle on tiny shapes drawn by hypothesis.

Each draw is checked against an enumeration written from the definitions,
independently of the oracle's C code:

- top-k (DeepSpeed #8195 change 3 and the Tutel gating it replaces): expert
  j is chosen iff fewer than k experts beat it, where i beats j when
  l_i > l_j, or l_i == l_j and i < j; its position is that number.
- the dispatch layout (the same change's location = cumsum - 1, GShard's
  k-major priority as the alternative order, Automodel #3684's per-expert
  padding, DeepSpeed #8213's per-rank dedup counts): walk the routes in
  priority order and hand each expert's next slot to the next route that
  names it; capacity keeps the first c; dropless rows are the exclusive
  scan of the (padded) counts plus the slot; a token counts once for each
  virtual rank that receives one of its kept routes, and its send slot is
  the number of earlier tokens that send to that rank.
- dispatch, combine and both backwards (the same change's gather and
  weighted combine; a backward is the other op with the gates applied or
  dropped): the dense one-hot route mask over the layout's rows, in
  float64.

The draws cover the degenerate cases the fixed pins do not enumerate: no
tokens, one expert, k = e, capacity 1, a pad larger than every segment,
one token per rank.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = dict(max_examples=300, deadline=None, derandomize=True)


@st.composite
def routing(draw):
    e = draw(st.integers(1, 8))
    k = draw(st.integers(1, e))
    s = draw(st.integers(0, 12))
    rows = [draw(st.permutations(list(range(e))))[:k] for _ in range(s)]
    idx = np.array(rows, np.int32).reshape(s, k)
    divisors = [r for r in range(1, e + 1) if e % r == 0]
    R = draw(st.sampled_from([0] + divisors))
    return idx, e, R


def enumerate_layout(idx, e, cap, R, kmajor, P):
    s, k = idx.shape
    order = [(t, j) for j in range(k) for t in range(s)] if kmajor else [(t, j) for t in range(s) for j in range(k)]
    loc = np.zeros((s, k), np.int64)
    taken = [0] * e
    for t, j in order:
        x = int(idx[t, j])
        loc[t, j] = taken[x]
        taken[x] += 1
    raw = np.array(taken, np.int64)
    drop = loc >= cap if cap else np.zeros((s, k), bool)
    counts = np.minimum(raw, cap) if cap else raw
    if cap:
        offsets = np.arange(e + 1, dtype=np.int64) * cap
        row = idx.astype(np.int64) * cap + loc
    else:
        seg = (counts + P - 1) // P * P
        offsets = np.concatenate([[0], np.cumsum(seg)]).astype(np.int64)
        row = offsets[idx] + loc if s else np.zeros((0, k), np.int64)
    row = np.where(drop, -1, row)
    out = dict(loc=loc, row=row, drop=drop, raw_counts=raw, counts=counts, offsets=offsets)
    if R:
        per = e // R
        tir = np.zeros((s, R), np.uint8)
        for t in range(s):
            for j in range(k):
                if not drop[t, j]:
                    tir[t, int(idx[t, j]) // per] = 1
        slot = np.full((s, R), -1, np.int64)
        for r in range(R):
            n = 0
            for t in range(s):
                if tir[t, r]:
                    slot[t, r] = n
                    n += 1
        out.update(token_in_rank=tir, rank_counts=tir.sum(0), rank_slot=slot)
    return out


@settings(**SETTINGS)
@given(routing(), st.integers(0, 5), st.booleans(), st.sampled_from([1, 2, 4, 16]))
def test_layout_matches_enumeration(r, cap, kmajor, P):
    idx, e, R = r
    if cap:
        P = 1  # padding applies to the dropless layout only
    L = oracle.layout(idx, e, cap, R, priority=1 if kmajor else 0, pad_multiple=P)
    want = enumerate_layout(idx, e, cap, R, kmajor, P)
    for name in ("loc", "row", "raw_counts", "counts", "offsets"):
        np.testing.assert_array_equal(L[name], want[name], err_msg=name)
    np.testing.assert_array_equal(L["drop"].astype(bool), want["drop"], err_msg="drop")
    assert L["rows"] == (e * cap if cap else idx.size + e * (P - 1))
    if R:
        for name in ("token_in_rank", "rank_counts", "rank_slot"):
            np.testing.assert_array_equal(L[name], want[name], err_msg=name)


@settings(**SETTINGS)
@given(st.integers(1, 8).flatmap(lambda e: st.tuples(
    st.just(e), st.integers(1, e),
    st.lists(st.lists(st.integers(-2, 2), min_size=e, max_size=e), min_size=1, max_size=6))))
def test_topk_matches_enumeration_with_many_ties(draw):
    e, k, rows = draw
    logits = np.array(rows, np.float32) * np.float32(0.5)  # small grid: ties everywhere
    idx, gate = oracle.topk_gate(logits, k)
    for t, l in enumerate(logits):
        want = np.full(k, -1)
        for j in range(e):
            beaten_by = sum(1 for i in range(e) if l[i] > l[j] or (l[i] == l[j] and i < j))
            if beaten_by < k:
                want[beaten_by] = j
        np.testing.assert_array_equal(idx[t], want)
    np.testing.assert_allclose(gate.sum(1), 1.0, rtol=1e-6)


@settings(**dict(SETTINGS, max_examples=150))
@given(routing(), st.integers(0, 5), st.booleans(), st.sampled_from([1, 4]), st.integers(1, 6),
       st.integers(0, 2**32 - 1))
def test_payload_ops_match_dense_route_masks(r, cap, kmajor, P, m, seed):
    """dispatch, combine and both backwards, fp32, on any layout variant:
    against the dense one-hot route mask M[t, row] (and its gate-weighted
    twin) in float64 -- X = M^T x, out = G y, dY = G^T dout, dgate[t, j] =
    <dout[t], y[row]>, dx = M dX; rows no route owns stay zero."""
    idx, e, R = r
    if cap:
        P = 1
    L = oracle.layout(idx, e, cap, R, priority=1 if kmajor else 0, pad_multiple=P)
    s, k = idx.shape
    rows = L["rows"]
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((s, m)).astype(np.float32)
    y = rng.standard_normal((rows, m)).astype(np.float32)
    dout = rng.standard_normal((s, m)).astype(np.float32)
    dX = rng.standard_normal((rows, m)).astype(np.float32)
    gate = (rng.random((s, k)) + 0.05).astype(np.float32)
    M = np.zeros((s, rows))
    G = np.zeros((s, rows))
    for t in range(s):
        for j in range(k):
            if not L["drop"][t, j]:
                M[t, L["row"][t, j]] = 1.0
                G[t, L["row"][t, j]] = float(gate[t, j])
    x64, y64, d64, dX64 = (a.astype(np.float64) for a in (x, y, dout, dX))

    X = oracle.dispatch(L["row"], x, rows)
    np.testing.assert_array_equal(X.astype(np.float64), M.T @ x64)

    out = oracle.combine(L["row"], gate, y).astype(np.float64)
    assert np.all(np.abs(out - G @ y64) <= 1e-6 * (G @ np.abs(y64)) + 1e-30)

    dY, dgate = oracle.combine_bwd(L["row"], gate, dout, y)
    ref = G.T @ d64
    assert np.all(np.abs(dY.astype(np.float64) - ref) <= 1e-6 * np.abs(ref) + 1e-30)
    for t in range(s):
        for j in range(k):
            if L["drop"][t, j]:
                assert dgate[t, j] == 0.0
            else:
                rr = L["row"][t, j]
                want = float(d64[t] @ y64[rr])
                assert abs(dgate[t, j] - want) <= 1e-6 * float(np.abs(d64[t]) @ np.abs(y64[rr])) + 1e-30

    dx = oracle.dispatch_bwd(L["row"], dX).astype(np.float64)
    assert np.all(np.abs(dx - M @ dX64) <= 1e-6 * (M @ np.abs(dX64)) + 1e-30)
