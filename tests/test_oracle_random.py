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
