"""NumPy front-end to the CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product package
never imports this module, and this module imports nothing from it.

Arrays are NumPy, C-contiguous; bf16 tensors travel as ``np.uint16`` bit
patterns.  Every function raises ``OracleError`` when the C code reports a
contract violation (see ``oracle.h``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
_ERRORS = {-1: "bad argument", -2: "non-finite logit", -3: "expert id out of range or repeated in a token"}


class OracleError(RuntimeError):
    pass


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L.ora_set_threads.argtypes = [I]
        L.ora_set_threads.restype = I
        L.ora_get_threads.restype = I
        L.ora_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_f32.restype = ctypes.c_float
        L.ora_f32_to_bf16.argtypes = [ctypes.c_float]
        L.ora_f32_to_bf16.restype = ctypes.c_uint16
        L.ora_topk_gate.argtypes = [P, I, I, I, I, P, P]
        L.ora_layout.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P, P, P]
        L.ora_topk_gate_bwd.argtypes = [P, P, P, P, I, I, I, I, P]
        L.ora_layout_ex.argtypes = [P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
        L.ora_dispatch.argtypes = [P, I, I, I, I, P, I, P]
        L.ora_combine.argtypes = [P, P, I, I, I, I, P, P]
        L.ora_combine_bwd.argtypes = [P, P, I, I, I, I, P, P, I, P, P]
        L.ora_dispatch_bwd.argtypes = [P, I, I, I, I, P, P]
        L.ora_rank_slots.argtypes = [P, I, I, P]
        for f in ("ora_topk_gate", "ora_topk_gate_bwd", "ora_layout", "ora_layout_ex", "ora_dispatch", "ora_combine",
                  "ora_combine_bwd", "ora_dispatch_bwd", "ora_rank_slots"):
            getattr(L, f).restype = I
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: {_ERRORS.get(rc, rc)}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle payloads are float32 or bf16-as-uint16, got {a.dtype}")


def set_threads(n: int) -> int:
    return lib().ora_set_threads(int(n))


def bf16_to_f32(b: int) -> float:
    return lib().ora_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return lib().ora_f32_to_bf16(float(f))


def topk_gate(logits: np.ndarray, k: int, renorm: int = 1):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    s, e = logits.shape
    idx = np.empty((s, k), np.int32)
    gate = np.empty((s, k), np.float32)
    _check(lib().ora_topk_gate(_p(logits), s, e, k, int(renorm), _p(idx), _p(gate)), "topk_gate")
    return idx, gate


def topk_gate_bwd(logits: np.ndarray | None, idx: np.ndarray, gate: np.ndarray, dgate: np.ndarray,
                  e: int, renorm: int = 1) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    dgate = np.ascontiguousarray(dgate, dtype=np.float32)
    lg = None if logits is None else np.ascontiguousarray(logits, dtype=np.float32)
    s, k = idx.shape
    dl = np.empty((s, e), np.float32)
    rc = lib().ora_topk_gate_bwd(_p(lg), _p(idx), _p(gate), _p(dgate), s, e, k, int(renorm), _p(dl))
    _check(rc, "topk_gate_bwd")
    return dl


def layout(idx: np.ndarray, e: int, capacity: int = 0, R: int = 0, priority: int = 0, pad_multiple: int = 1) -> dict:
    """Dispatch layout; priority 0 = token order, 1 = k-major; pad_multiple
    pads each expert's dropless rows to a multiple (rows is then the upper
    bound s*k + e*(pad_multiple - 1))."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    s, k = idx.shape
    out = dict(
        loc=np.empty((s, k), np.int32), row=np.empty((s, k), np.int32), drop=np.empty((s, k), np.uint8),
        raw_counts=np.empty(e, np.int32), counts=np.empty(e, np.int32), offsets=np.empty(e + 1, np.int32),
        token_in_rank=np.empty((s, R), np.uint8) if R else None,
        rank_counts=np.empty(R, np.int32) if R else None,
    )
    rc = lib().ora_layout_ex(_p(idx), s, e, k, int(capacity), int(R), int(priority), int(pad_multiple),
                             _p(out["loc"]), _p(out["row"]), _p(out["drop"]), _p(out["raw_counts"]),
                             _p(out["counts"]), _p(out["offsets"]), _p(out["token_in_rank"]),
                             _p(out["rank_counts"]))
    _check(rc, "layout")
    out["rows"] = e * capacity if capacity > 0 else s * k + e * (pad_multiple - 1)
    out["rank_slot"] = rank_slots(out["token_in_rank"]) if R else None
    return out


def rank_slots(token_in_rank: np.ndarray) -> np.ndarray:
    """Token-order send slot of each token in each virtual rank it sends to
    (-1 where it sends nothing); token_in_rank [s, R] from layout()."""
    tir = np.ascontiguousarray(token_in_rank, dtype=np.uint8)
    s, R = tir.shape
    out = np.empty((s, R), np.int32)
    _check(lib().ora_rank_slots(_p(tir), s, R, _p(out)), "rank_slots")
    return out


def dispatch(row: np.ndarray, x: np.ndarray, rows: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.int32)
    x = np.ascontiguousarray(x)
    s, k = row.shape
    m = x.shape[1]
    X = np.empty((rows, m), x.dtype)
    _check(lib().ora_dispatch(_p(row), s, k, m, _dtype_code(x), _p(x), rows, _p(X)), "dispatch")
    return X


def combine(row: np.ndarray, gate: np.ndarray | None, y: np.ndarray) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.int32)
    y = np.ascontiguousarray(y)
    s, k = row.shape
    m = y.shape[1]
    g = None if gate is None else np.ascontiguousarray(gate, dtype=np.float32)
    out = np.empty((s, m), y.dtype)
    _check(lib().ora_combine(_p(row), _p(g), s, k, m, _dtype_code(y), _p(y), _p(out)), "combine")
    return out


def combine_bwd(row: np.ndarray, gate: np.ndarray, dout: np.ndarray, y: np.ndarray):
    row = np.ascontiguousarray(row, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    dout = np.ascontiguousarray(dout)
    y = np.ascontiguousarray(y)
    assert dout.dtype == y.dtype
    s, k = row.shape
    m = dout.shape[1]
    rows = y.shape[0]
    dY = np.empty((rows, m), dout.dtype)
    dgate = np.empty((s, k), np.float32)
    rc = lib().ora_combine_bwd(_p(row), _p(gate), s, k, m, _dtype_code(dout), _p(dout), _p(y), rows,
                               _p(dY), _p(dgate))
    _check(rc, "combine_bwd")
    return dY, dgate


def dispatch_bwd(row: np.ndarray, dX: np.ndarray) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.int32)
    dX = np.ascontiguousarray(dX)
    s, k = row.shape
    m = dX.shape[1]
    dx = np.empty((s, m), dX.dtype)
    _check(lib().ora_dispatch_bwd(_p(row), s, k, m, _dtype_code(dX), _p(dX), _p(dx)), "dispatch_bwd")
    return dx


def grouped_gemm(X: np.ndarray, W: np.ndarray, offsets: np.ndarray, counts: np.ndarray) -> np.ndarray:
    """Y[r] = X[r] . W[x]^T in float64 for the rows a route owns (the first
    counts[x] rows of expert x's segment); other rows NaN.  X [rows,K] and W
    [e,N,K] as float32 or bf16-as-uint16.  One library matmul per expert."""
    def f64(a):
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if a.dtype == np.uint16 \
            else a.astype(np.float64)
    Xf, Wf = f64(X), f64(W)
    Y = np.full((X.shape[0], W.shape[1]), np.nan)
    for x in range(W.shape[0]):
        r0, n = int(offsets[x]), int(counts[x])
        if n:
            Y[r0:r0 + n] = Xf[r0:r0 + n] @ Wf[x].T
    return Y
