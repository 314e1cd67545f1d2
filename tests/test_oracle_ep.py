"""Pins of the expert-parallel oracle (``oracle/ep.py``) against things
other than itself: with one rank it must be the single-GPU path bit for
bit; for any rank count, the dedup and conservation the page states
(DeepSpeed #8213, description: a token goes to each destination rank once,
not once per selected expert), the expert grouping checked by enumeration,
agreement with the single-GPU combine up to the extra rounding the per-rank
partials add, and the adjoint identities of the forward and backward pairs.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import ep
from combine_moe_topk_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def expert(X: np.ndarray, expert_of_row: np.ndarray) -> np.ndarray:
    """An exact, expert-dependent output: row times 2^((x % 3) - 1)."""
    scale = np.float32(2.0) ** ((expert_of_row % 3) - 1).astype(np.float32)
    if X.dtype == np.uint16:
        f = (X.astype(np.uint32) << 16).view(np.float32) * scale[:, None]
        return (f.view(np.uint32) >> 16).astype(np.uint16)  # exact: a power-of-two scale
    return (X * scale[:, None]).astype(np.float32)


def expert_rows(offsets, counts, rows, e_offset=0):
    ex = np.full(rows, -1, np.int64)
    for x in range(len(counts)):
        ex[offsets[x]:offsets[x] + counts[x]] = x + e_offset
    return ex


def rank_inputs(R, s, m, e, k, dtype, seed, zipf=0.0):
    xs, idxs, gates = [], [], []
    for r in range(R):
        w = W.Workload("ep", s=s, m=m, e=e, k=k, dtype=dtype, capacity=0, R=R, seed=seed + r, zipf_alpha=zipf)
        inp = W.make_inputs(w, with_grad=False)
        idx, gate = oracle.topk_gate(inp["logits"].numpy(), k, 1)
        if dtype == "bf16":
            x = inp["x"].contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            x = inp["x"].numpy()
        xs.append(x)
        idxs.append(idx)
        gates.append(gate)
    return xs, idxs, gates


def local_outputs(st):
    return [expert(st["X"][d], expert_rows(st["locs"][d]["offsets"], st["locs"][d]["counts"], st["locs"][d]["rows"],
                                           d * st["E"])) for d in range(st["R"])]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_rank_is_the_single_gpu_path(dtype):
    s, m, e, k = 300, 16, 8, 2
    xs, idxs, gates = rank_inputs(1, s, m, e, k, dtype, seed=1)
    st = ep.ep_dispatch(xs, idxs, gates, e, 1)
    L = oracle.layout(idxs[0], e, 0, 1)
    X = oracle.dispatch(L["row"], xs[0], L["rows"])
    np.testing.assert_array_equal(st["X"][0], X)
    ys = local_outputs(st)
    y = expert(X, expert_rows(L["offsets"], L["counts"], L["rows"]))
    np.testing.assert_array_equal(ys[0], y)
    np.testing.assert_array_equal(ep.ep_combine(st, ys)[0], oracle.combine(L["row"], gates[0], y))
    rng = np.random.default_rng(3)
    dout = rng.standard_normal((s, m)).astype(np.float32)
    if dtype == "bf16":
        dout = (dout.view(np.uint32) >> 16).astype(np.uint16)
    dY, dg = ep.ep_combine_bwd(st, [dout], ys)
    OdY, Odg = oracle.combine_bwd(L["row"], gates[0], dout, y)
    np.testing.assert_array_equal(dY[0], OdY)
    np.testing.assert_array_equal(dg[0], Odg)
    np.testing.assert_array_equal(ep.ep_dispatch_bwd(st, dY)[0], oracle.dispatch_bwd(L["row"], OdY))


@pytest.mark.parametrize("R", [2, 4, 8])
def test_each_token_goes_to_each_rank_once_and_every_route_arrives(R):
    """Dedup and conservation, by enumeration: rank d receives token t of
    source r exactly once iff one of t's routes goes to an expert of d; the
    arrivals total the sum of the sources' rank counts; each local expert's
    rows are the rows of the routes to it, in (source, token) order."""
    s, m, e, k = 200, 8, 16, 4
    xs, idxs, gates = rank_inputs(R, s, m, e, k, "f32", seed=10, zipf=1.0)
    st = ep.ep_dispatch(xs, idxs, gates, e, R)
    E = e // R
    assert sum(len(st["recv_x"][d]) for d in range(R)) == int(st["counts"].sum())
    for d in range(R):
        want = [(r, t) for r in range(R) for t in range(s) if any(idxs[r][t, j] // E == d for j in range(k))]
        assert len(st["recv_x"][d]) == len(want)
        for i, (r, t) in enumerate(want):
            np.testing.assert_array_equal(st["recv_x"][d][i], xs[r][t])
            for j in range(k):
                x = idxs[r][t, j]
                assert st["recv_idx"][d][i, j] == (x - d * E if x // E == d else -1)
                assert st["recv_gate"][d][i, j] == (gates[r][t, j] if x // E == d else 0)
        loc = st["locs"][d]
        for x in range(E):
            rows = [xs[r][t] for r in range(R) for t in range(s) for j in range(k) if idxs[r][t, j] == d * E + x]
            seg = st["X"][d][loc["offsets"][x]:loc["offsets"][x] + loc["counts"][x]]
            assert len(seg) == len(rows)
            if rows:
                np.testing.assert_array_equal(seg, np.stack(rows))
    # each token counted once per destination: never more arrivals than routes
    routes_per_rank = [[sum(1 for t in range(s) for j in range(k) if idxs[r][t, j] // E == d) for d in range(R)]
                       for r in range(R)]
    assert np.all(st["counts"] <= np.array(routes_per_rank))


@pytest.mark.parametrize("R", [2, 4])
def test_capacity_drops_are_not_sent(R):
    s, m, e, k, cap = 120, 8, 8, 2, 20
    xs, idxs, gates = rank_inputs(R, s, m, e, k, "f32", seed=20, zipf=1.5)
    st = ep.ep_dispatch(xs, idxs, gates, e, R, capacity=cap)
    E = e // R
    for r in range(R):
        L = oracle.layout(idxs[r], e, cap, R)
        assert L["drop"].any()
        for d in range(R):
            kept = [t for t in range(s) if any(L["row"][t, j] >= 0 and idxs[r][t, j] // E == d for j in range(k))]
            assert st["counts"][r, d] == len(kept)


@pytest.mark.parametrize("R", [2, 4, 8])
def test_fp32_agrees_with_the_single_gpu_combine(R):
    """Per-rank partials change only the association of the fp32 sum: within
    1e-6 of the condition scale sum_j |g_j| |y_j| of the one-GPU combine of
    the same expert outputs."""
    s, m, e, k = 150, 12, 16, 4
    xs, idxs, gates = rank_inputs(R, s, m, e, k, "f32", seed=30)
    st = ep.ep_dispatch(xs, idxs, gates, e, R)
    out = ep.ep_combine(st, local_outputs(st))
    for r in range(R):
        L = oracle.layout(idxs[r], e, 0, 0)
        X = oracle.dispatch(L["row"], xs[r], L["rows"])
        y = expert(X, expert_rows(L["offsets"], L["counts"], L["rows"]))
        single = oracle.combine(L["row"], gates[r], y).astype(np.float64)
        scale = np.zeros((s, m))
        for j in range(k):
            scale += np.abs(gates[r][:, j:j + 1].astype(np.float64)) * np.abs(y[L["row"][:, j]].astype(np.float64))
        assert np.all(np.abs(out[r] - single) <= 1e-6 * scale + 1e-30)


def test_adjoint_identities():
    """<ep_dispatch(x), dX> = <x, ep_dispatch_bwd(dX)> and
    <ep_combine(y), dout> = <y, dY> over all ranks, in float64 (fp32 data,
    one-rounding bounds)."""
    R, s, m, e, k = 4, 100, 8, 16, 3
    xs, idxs, gates = rank_inputs(R, s, m, e, k, "f32", seed=40)
    st = ep.ep_dispatch(xs, idxs, gates, e, R)
    rng = np.random.default_rng(5)
    dX = [rng.standard_normal(X.shape).astype(np.float32) for X in st["X"]]
    dx = ep.ep_dispatch_bwd(st, dX)
    lhs = sum(float(np.sum(st["X"][d].astype(np.float64) * dX[d])) for d in range(R))
    rhs = sum(float(np.sum(xs[r].astype(np.float64) * dx[r])) for r in range(R))
    assert abs(lhs - rhs) <= 1e-5 * (abs(lhs) + 1)
    ys = [rng.standard_normal(X.shape).astype(np.float32) for X in st["X"]]
    douts = [rng.standard_normal((s, m)).astype(np.float32) for _ in range(R)]
    out = ep.ep_combine(st, ys)
    dY, dgate = ep.ep_combine_bwd(st, douts, ys)
    lhs = sum(float(np.sum(out[r].astype(np.float64) * douts[r])) for r in range(R))
    rhs = sum(float(np.sum(ys[d].astype(np.float64) * dY[d])) for d in range(R))
    assert abs(lhs - rhs) <= 1e-5 * (abs(lhs) + 1)
    # the gate gradient of a route is the dot of its token's upstream
    # gradient with the expert output row of that route (a copy went out)
    E = e // R
    for r in range(R):
        L = oracle.layout(idxs[r], e, 0, R)
        for t in range(0, s, 7):
            for j in range(k):
                d = idxs[r][t, j] // E
                i = int(np.nonzero([(rr == r) for rr in
                                    [src for src in range(R) for _ in range(st["counts"][src, d])]])[0][0])
                i += int(st["plans"][r]["send_row"][t, d] - st["plans"][r]["send_off"][d])
                row = st["locs"][d]["row"][i, j]
                want = float(np.dot(douts[r][t].astype(np.float64), ys[d][row].astype(np.float64)))
                assert abs(dgate[r][t, j] - want) <= 1e-6 * (abs(want) + 1e-30) + 1e-12
