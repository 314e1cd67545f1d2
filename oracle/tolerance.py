"""Comparison rules between the CUDA path and the oracle (test infrastructure).

The bar, per output kind:
* integers, indices, bytes and copied rows: bit-exact;
* fp32 floating outputs of a reduction: |gpu - oracle| <= 1e-6 * scale + 1e-30,
  with scale the condition number's numerator, elementwise: sum_j |g_j|*|y_j|
  for a combine, sum_m |dout*y| for a gate gradient, |g|*|dout| for a scaled
  copy;
* bf16 outputs: within one bf16 ulp of the oracle's value;
* gates: relative 1e-6.
"""
from __future__ import annotations

import numpy as np

REL_F32 = 1e-6


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-126)))
    return 2.0 ** (e - 7)


def combine_scale(row: np.ndarray, gate: np.ndarray | None, y: np.ndarray) -> np.ndarray:
    """sum over kept routes of |gate| * |y[row]|, float64 [s, m]."""
    s, k = row.shape
    out = np.zeros((s, y.shape[1]))
    for j in range(k):
        r = row[:, j]
        keep = r >= 0
        g = np.ones(s) if gate is None else np.abs(gate[:, j].astype(np.float64))
        out[keep] += g[keep, None] * np.abs(as_f64(y[r[keep]]))
    return out


def dot_scale(row: np.ndarray, dout: np.ndarray, y: np.ndarray) -> np.ndarray:
    """sum_m |dout[t,m] * y[row[t,j],m]|, float64 [s, k]."""
    s, k = row.shape
    da = np.abs(as_f64(dout))
    out = np.zeros((s, k))
    for j in range(k):
        r = row[:, j]
        keep = r >= 0
        out[keep, j] = np.sum(da[keep] * np.abs(as_f64(y[r[keep]])), axis=1)
    return out


def gate_bwd_scale(idx: np.ndarray, gate: np.ndarray, dgate_scale: np.ndarray, e: int, renorm: int,
                   logits: np.ndarray | None = None) -> np.ndarray:
    """Condition scale of the gate backward per logit, float64 [s, e]:
    fac_i * (dgate_scale(i) + sum_j |g_j| dgate_scale_j), fac = the gate of
    a selected expert (renorm) or the full-softmax probability (no renorm).
    dgate_scale is |dgate| for an op-level check, or the upstream gate
    gradient's own scale when dgate was computed in floating point."""
    s, k = idx.shape
    ii = idx.astype(np.int64)
    ds = np.abs(np.asarray(dgate_scale, np.float64))
    c = np.sum(np.abs(gate.astype(np.float64)) * ds, axis=1, keepdims=True)
    dg = np.zeros((s, e))
    np.put_along_axis(dg, ii, ds, 1)
    if renorm:
        fac = np.zeros((s, e))
        np.put_along_axis(fac, ii, np.abs(gate.astype(np.float64)), 1)
    else:
        l = logits.astype(np.float64)
        p = np.exp(l - l.max(axis=1, keepdims=True))
        fac = p / p.sum(axis=1, keepdims=True)
    return fac * (dg + c)


def assert_close(gpu: np.ndarray, ora: np.ndarray, scale, what: str):
    """Apply the rule for the array's type (uint16 = bf16 bits, float32).

    ``scale`` is the float64 condition scale of every element, or a function
    of an array of first-axis indices returning the scale of those rows
    only: then it is evaluated just for the rows that are not bit-identical
    (the same bar, without building the scale of a multi-GB array whose
    elements mostly match exactly)."""
    assert gpu.shape == ora.shape, f"{what}: shape {gpu.shape} vs {ora.shape}"
    if np.array_equal(gpu, ora):
        return
    rows = None
    if callable(scale):
        diff = gpu != ora
        rows = np.unique(np.nonzero(diff.reshape(diff.shape[0], -1))[0])
        gpu, ora, scale = gpu[rows], ora[rows], (None if ora.dtype == np.uint16 else scale(rows))
    g, o = as_f64(gpu), as_f64(ora)
    if ora.dtype == np.uint16:
        bad = ~(np.abs(g - o) <= bf16_ulp(o))
    else:
        assert scale is not None
        bad = ~(np.abs(g - o) <= REL_F32 * scale + 1e-30)
    if bad.any():
        i = tuple(int(v) for v in np.argwhere(bad)[0])
        at = i if rows is None else (int(rows[i[0]]),) + i[1:]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {at}: "
                             f"gpu {g[i]!r} oracle {o[i]!r}")


def assert_gates_close(gpu: np.ndarray, ora: np.ndarray, what: str = "gate"):
    err = np.abs(gpu.astype(np.float64) - ora.astype(np.float64))
    bad = err > REL_F32 * np.abs(ora.astype(np.float64))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} gates off by more than 1e-6 relative; first at {i}: "
                             f"gpu {gpu[i]!r} oracle {ora[i]!r}")
