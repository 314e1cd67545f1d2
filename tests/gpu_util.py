"""Shared helpers of the GPU parity tests: moving arrays between torch and
NumPy (bf16 as uint16 bit patterns), and running the whole path once on the
GPU and once in the oracle on identical inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import tolerance as T
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


LAYOUT_FIELDS = ("idx", "loc", "row", "drop", "raw_counts", "counts", "offsets")


def check_layout(h: B.Handle, L: dict, idx: np.ndarray):
    got = {n: bits(getattr(h, n)()) for n in LAYOUT_FIELDS}
    np.testing.assert_array_equal(got["idx"], idx, err_msg="idx copy")
    for n in LAYOUT_FIELDS[1:]:
        np.testing.assert_array_equal(got[n], L[n], err_msg=n)
    if h.R:
        np.testing.assert_array_equal(bits(h.token_in_rank()), L["token_in_rank"], err_msg="token_in_rank")
        np.testing.assert_array_equal(bits(h.rank_counts()), L["rank_counts"], err_msg="rank_counts")


def full_parity(w, dev, renorm=None, seed=None, priority="token", pad_multiple=1):
    """Run gate -> layout -> dispatch -> combine -> combine_bwd -> dispatch_bwd
    on the GPU and in the oracle on the same seeded inputs; compare all.
    priority / pad_multiple select a layout variant (moe_dispatch_layout_ex)."""
    renorm = w.renorm if renorm is None else renorm
    if pad_multiple > 1:
        w = w.replace(capacity=0)
    # a padded layout's buffer has e * (pad_multiple - 1) more rows than the workload's
    rows = w.rows + (w.e * (pad_multiple - 1) if pad_multiple > 1 else 0)
    inp = W.make_inputs(w, seed=seed, rows=rows)
    g = {k: v.to(dev) for k, v in inp.items()}

    # gate
    idx, gate = B.moe_topk_gate(g["logits"], w.k, renorm)
    oi, og = oracle.topk_gate(inp["logits"].numpy(), w.k, renorm)
    np.testing.assert_array_equal(bits(idx), oi, err_msg="topk idx")
    T.assert_gates_close(bits(gate), og)

    # layout on the oracle's ids (equal to the GPU's, asserted above)
    if priority == "token" and pad_multiple == 1:
        h = B.moe_dispatch_layout(to_dev(oi, dev), w.e, w.capacity, w.R)
    else:
        h = B.moe_dispatch_layout_ex(to_dev(oi, dev), w.e, w.capacity, w.R, priority, pad_multiple)
    L = oracle.layout(oi, w.e, w.capacity, w.R, priority=1 if priority == "kmajor" else 0,
                      pad_multiple=pad_multiple)
    assert h.rows == L["rows"]
    check_layout(h, L, oi)
    row = L["row"]

    # dispatch: a copy, bit-exact
    xb = bits(inp["x"])
    X = B.moe_dispatch(h, g["x"])
    np.testing.assert_array_equal(bits(X), oracle.dispatch(row, xb, L["rows"]), err_msg="dispatch")

    # combine with the oracle's gates on both sides
    gd = to_dev(og, dev)
    yb, db = bits(inp["y"]), bits(inp["dout"])
    out = B.moe_combine(h, g["y"], gd)
    T.assert_close(bits(out), oracle.combine(row, og, yb), T.combine_scale(row, og, yb), "combine")

    dY, dgate = B.moe_combine_bwd(h, g["dout"], gd, g["y"])
    OdY, Odg = oracle.combine_bwd(row, og, db, yb)
    T.assert_close(bits(dY), OdY, np.abs(T.as_f64(OdY)), "dY")
    T.assert_close(bits(dgate), Odg, T.dot_scale(row, db, yb), "dgate")

    dx = B.moe_dispatch_bwd(h, to_dev(OdY, dev))
    T.assert_close(bits(dx), oracle.dispatch_bwd(row, OdY), T.combine_scale(row, None, OdY), "dx")
    assert h.status() == 0
    return h, L
