"""ctypes binding of ``libmoe_gb300.so`` (C ABI in ``include/moe_gb300.h``).

Argument marshalling only: every step of the token path runs in the CUDA
library.  PyTorch supplies device memory (outputs are allocated with
``torch.empty`` when the caller does not pass them) and the current CUDA
stream.  The functions keep the C names; tensors replace (pointer, size)
pairs.  Every non-OK status raises ``MoEError``; if the shared library is
missing the first call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_DTYPE",
    4: "MOE_ERR_HANDLE_MISMATCH", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_OOM", 7: "MOE_ERR_TIMEOUT",
    8: "MOE_ERR_NONFINITE", 9: "MOE_ERR_BAD_ROUTE",
}
MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
MOE_DEV_NONFINITE, MOE_DEV_BAD_ROUTE, MOE_DEV_TIMEOUT, MOE_DEV_ROWS_EXCEEDED = 0x1, 0x2, 0x4, 0x8
KERNELS = ["topk_gate", "layout", "dispatch", "combine", "combine_bwd", "dispatch_bwd", "topk_gate_bwd",
           "grouped_gemm", "dispatch_gemm", "rank_slots", "combine_gate_bwd", "gate_layout", "ep_pack", "ep_unpack",
           "ep_dispatch", "ep_combine"]
KERNEL_ID = {n: i for i, n in enumerate(KERNELS)}

# every entry point the header declares (checked by the CPU test-suite)
EXPORTS = [
    "moe_topk_gate", "moe_dispatch_layout", "moe_dispatch", "moe_combine", "moe_combine_bwd",
    "moe_dispatch_bwd", "moe_handle_info", "moe_handle_status", "moe_handle_destroy", "moe_capacity",
    "moe_status_string", "moe_last_error", "moe_launch_count", "moe_debug_hold_layout_tile",
    "moe_dispatch_layout_noalloc", "moe_topk_gate_bwd", "moe_dispatch_layout_ex", "moe_grouped_gemm",
    "moe_dispatch_grouped_gemm", "moe_combine_gate_bwd", "moe_layout_create", "moe_layout_rebuild",
    "moe_topk_gate_layout", "moe_ep_pack", "moe_ep_dispatch", "moe_ep_combine", "moe_ep_unpack_dgate",
]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name}" + (f" ({detail})" if detail else ""))


class LayoutOptions(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int32), ("num_virtual_ranks", ctypes.c_int32), ("priority", ctypes.c_int32),
                ("pad_multiple", ctypes.c_int32), ("send_slots", ctypes.c_int32), ("absent_routes", ctypes.c_int32),
                ("rows_bound", ctypes.c_int32)]


PRIORITY = {"token": 0, "kmajor": 1}


class LayoutInfo(ctypes.Structure):
    _fields_ = [("s", ctypes.c_int32), ("e", ctypes.c_int32), ("k", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("R", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("device", ctypes.c_int32), ("priority", ctypes.c_int32), ("pad_multiple", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("idx", "loc", "row", "drop", "raw_counts", "counts", "offsets",
                                       "token_in_rank", "rank_counts", "status", "inv_row", "rank_slot")]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                               "g.build()\"` (nvcc, sm_103a); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, I, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
        sig = {
            "moe_topk_gate": [P, I, I, I, I, P, P, P, P],
            "moe_topk_gate_bwd": [P, P, P, P, I, I, I, I, P, P],
            "moe_dispatch_layout": [P, I, I, I, I, I, P, ctypes.POINTER(P)],
            "moe_dispatch_layout_ex": [P, I, I, I, ctypes.POINTER(LayoutOptions), P, ctypes.POINTER(P)],
            "moe_layout_create": [I, I, I, ctypes.POINTER(LayoutOptions), P, ctypes.POINTER(P)],
            "moe_layout_rebuild": [P, P, P],
            "moe_topk_gate_layout": [P, P, I, P, P, P],
            "moe_ep_pack": [P, P, I, P, P, P, P],
            "moe_ep_dispatch": [P, P, I, I, I, P, P, P],
            "moe_ep_combine": [P, P, I, I, I, P, P, P],
            "moe_ep_unpack_dgate": [P, P, I, P, P, P],
            "moe_dispatch": [P, I, I, I, I, P, P, P],
            "moe_combine": [P, I, I, I, I, P, P, P, P],
            "moe_combine_bwd": [P, I, I, I, I, P, P, P, P, P, P],
            "moe_combine_gate_bwd": [P, I, I, I, I, P, P, P, P, I, P, P, P, P],
            "moe_dispatch_bwd": [P, I, I, I, I, P, P, P],
            "moe_grouped_gemm": [P, I, I, I, P, P, P, P],
            "moe_dispatch_grouped_gemm": [P, I, I, I, I, P, P, P, P],
            "moe_handle_info": [P, ctypes.POINTER(LayoutInfo)],
            "moe_handle_status": [P, P, ctypes.POINTER(ctypes.c_int32)],
            "moe_handle_destroy": [P],
            "moe_debug_hold_layout_tile": [I, I],
            "moe_dispatch_layout_noalloc": [P, I, I, I, I, I] + [P] * 11,
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = I
        L.moe_capacity.argtypes = [ctypes.c_double, I, I, I]
        L.moe_capacity.restype = I
        L.moe_status_string.argtypes = [I]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_launch_count.argtypes = [I]
        L.moe_launch_count.restype = U
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != MOE_OK:
        detail = lib().moe_last_error().decode(errors="replace")
        raise MoEError(rc, where, detail)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _stream(device: torch.device):
    # a host tensor still goes to the library, which rejects it; use the current device's stream
    dev = device if device.type == "cuda" else None
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float16:
        return MOE_F16
    return -1


# ------------------------------------------------------------------ handle --

class _DeviceArray:
    """A CUDA array view of handle memory (``__cuda_array_interface__``); treat it as read-only."""

    def __init__(self, owner, ptr: int, shape: tuple, typestr: str):
        self._owner = owner  # keeps the handle (and its memory) alive
        self.__cuda_array_interface__ = {
            "shape": shape, "typestr": typestr, "data": (ptr or 0, False), "version": 3, "strides": None,
            "stream": None,
        }


class Handle:
    """Owns a ``moe_handle``; destroys it when garbage-collected."""

    def __init__(self, raw: ctypes.c_void_p, device: torch.device):
        self._raw = raw
        self.device = device
        info = LayoutInfo()
        _check(lib().moe_handle_info(raw, ctypes.byref(info)), "moe_handle_info")
        self.info = info
        self.s, self.e, self.k = info.s, info.e, info.k
        self.capacity, self.R, self.rows = info.capacity, info.R, info.rows
        self.priority, self.pad_multiple = info.priority, info.pad_multiple

    @property
    def raw(self):
        if self._raw is None:
            raise MoEError(4, "handle", "destroyed")
        return self._raw

    def _view(self, name: str, shape: tuple, typestr: str) -> torch.Tensor:
        ptr = getattr(self.info, name)
        if not ptr or 0 in shape:
            dt = {"<i4": torch.int32, "|u1": torch.uint8}[typestr]
            return torch.empty(shape, dtype=dt, device=self.device)
        return torch.as_tensor(_DeviceArray(self, ptr, shape, typestr), device=self.device)

    # device arrays of the layout (views of handle memory, valid while the handle lives)
    def idx(self): return self._view("idx", (self.s, self.k), "<i4")
    def loc(self): return self._view("loc", (self.s, self.k), "<i4")
    def row(self): return self._view("row", (self.s, self.k), "<i4")
    def drop(self): return self._view("drop", (self.s, self.k), "|u1")
    def raw_counts(self): return self._view("raw_counts", (self.e,), "<i4")
    def counts(self): return self._view("counts", (self.e,), "<i4")
    def offsets(self): return self._view("offsets", (self.e + 1,), "<i4")
    def token_in_rank(self): return self._view("token_in_rank", (self.s, self.R), "|u1")
    def rank_counts(self): return self._view("rank_counts", (self.R,), "<i4")
    def inv_row(self): return self._view("inv_row", (self.rows,), "<i4")
    def rank_slot(self):
        if not self.info.rank_slot:
            raise MoEError(1, "rank_slot", "the handle was built without send_slots")
        return self._view("rank_slot", (self.s, self.R), "<i4")

    def status(self) -> int:
        """Synchronise and read the device status word (MOE_DEV_* bits)."""
        v = ctypes.c_int32(0)
        _check(lib().moe_handle_status(self.raw, _stream(self.device), ctypes.byref(v)), "moe_handle_status")
        return v.value

    def destroy(self):
        if self._raw is not None:
            raw, self._raw = self._raw, None
            with torch.cuda.device(self.device):
                _check(lib().moe_handle_destroy(raw), "moe_handle_destroy")

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


# ------------------------------------------------------------- entry points --

def moe_capacity(capacity_factor: float, s: int, k: int, e: int) -> int:
    return lib().moe_capacity(float(capacity_factor), int(s), int(k), int(e))


def moe_launch_count(kernel: str | int) -> int:
    return lib().moe_launch_count(KERNEL_ID.get(kernel, kernel) if isinstance(kernel, str) else kernel)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_debug_hold_layout_tile(tile: int, timeout_ms: int = 200):
    _check(lib().moe_debug_hold_layout_tile(int(tile), int(timeout_ms)), "moe_debug_hold_layout_tile")


def moe_topk_gate(logits: torch.Tensor, k: int, renorm: int = 1, topk_idx: torch.Tensor | None = None,
                  topk_gate: torch.Tensor | None = None, device_status: torch.Tensor | None = None):
    """logits f32 [s,e] -> (idx i32 [s,k], gate f32 [s,k])."""
    if logits.dim() != 2:
        raise ValueError("logits must be [s, e]")
    s, e = logits.shape
    if logits.dtype != torch.float32:
        raise MoEError(3, "moe_topk_gate", "logits must be float32")
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty(s, k, dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty(s, k, dtype=torch.float32, device=dev)
    rc = lib().moe_topk_gate(_ptr(logits), s, e, int(k), int(renorm), _ptr(topk_idx), _ptr(topk_gate),
                             _ptr(device_status), _stream(dev))
    _check(rc, "moe_topk_gate")
    return topk_idx, topk_gate


def moe_topk_gate_bwd(logits: torch.Tensor | None, topk_idx: torch.Tensor, topk_gate: torch.Tensor,
                      dgate: torch.Tensor, e: int, renorm: int = 1, dlogits: torch.Tensor | None = None):
    """(logits f32 [s,e] or None when renorm=1, idx [s,k], gate [s,k], dgate [s,k]) -> dlogits f32 [s,e]."""
    s, k = topk_idx.shape
    for t, name in ((topk_gate, "topk_gate"), (dgate, "dgate")):
        if t.dtype != torch.float32 or tuple(t.shape) != (s, k):
            raise MoEError(1, "moe_topk_gate_bwd", f"{name} must be float32 [s, k]")
    if logits is not None and (logits.dtype != torch.float32 or tuple(logits.shape) != (s, e)):
        raise MoEError(1, "moe_topk_gate_bwd", "logits must be float32 [s, e]")
    dev = topk_idx.device
    if dlogits is None:
        dlogits = torch.empty(s, e, dtype=torch.float32, device=dev)
    rc = lib().moe_topk_gate_bwd(_ptr(logits), _ptr(topk_idx), _ptr(topk_gate), _ptr(dgate), s, int(e), k,
                                 int(renorm), _ptr(dlogits), _stream(dev))
    _check(rc, "moe_topk_gate_bwd")
    return dlogits


def moe_dispatch_layout(topk_idx: torch.Tensor, e: int, capacity: int = 0, num_virtual_ranks: int = 0) -> Handle:
    """topk_idx i32 [s,k] -> Handle (counts, locations, rows, drops, dedup counts)."""
    if topk_idx.dim() != 2 or topk_idx.dtype != torch.int32:
        raise ValueError("topk_idx must be int32 [s, k]")
    s, k = topk_idx.shape
    raw = ctypes.c_void_p()
    dev = topk_idx.device
    rc = lib().moe_dispatch_layout(_ptr(topk_idx), s, int(e), k, int(capacity), int(num_virtual_ranks),
                                   _stream(dev), ctypes.byref(raw))
    _check(rc, "moe_dispatch_layout")
    return Handle(raw, dev)


def moe_dispatch_layout_ex(topk_idx: torch.Tensor, e: int, capacity: int = 0, num_virtual_ranks: int = 0,
                           priority: str = "token", pad_multiple: int = 1, send_slots: bool = False,
                           absent_routes: bool = False, rows_bound: int = 0) -> Handle:
    """Layout with a capacity priority ("token" or "kmajor"), per-expert
    padding of the dropless rows (handle.rows is then an upper bound),
    with send_slots each token's token-order slot per virtual rank
    (handle.rank_slot()), with absent_routes expert id -1 taken as a
    route that does not exist, and with rows_bound (dropless) the caller's
    bound on the kept routes as the handle's rows."""
    if topk_idx.dim() != 2 or topk_idx.dtype != torch.int32:
        raise ValueError("topk_idx must be int32 [s, k]")
    s, k = topk_idx.shape
    opt = LayoutOptions(int(capacity), int(num_virtual_ranks), PRIORITY[priority], int(pad_multiple),
                        int(bool(send_slots)), int(bool(absent_routes)), int(rows_bound))
    raw = ctypes.c_void_p()
    dev = topk_idx.device
    rc = lib().moe_dispatch_layout_ex(_ptr(topk_idx), s, int(e), k, ctypes.byref(opt), _stream(dev),
                                      ctypes.byref(raw))
    _check(rc, "moe_dispatch_layout_ex")
    return Handle(raw, dev)


def moe_layout_create(s: int, e: int, k: int, capacity: int = 0, num_virtual_ranks: int = 0,
                      priority: str = "token", pad_multiple: int = 1, send_slots: bool = False,
                      device: torch.device | None = None, absent_routes: bool = False,
                      rows_bound: int = 0) -> Handle:
    """An empty handle for [s, k] routes over e experts with these layout
    options, to be built (and rebuilt) in place by moe_layout_rebuild or
    moe_topk_gate_layout without allocating."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    opt = LayoutOptions(int(capacity), int(num_virtual_ranks), PRIORITY[priority], int(pad_multiple),
                        int(bool(send_slots)), int(bool(absent_routes)), int(rows_bound))
    raw = ctypes.c_void_p()
    with torch.cuda.device(dev):
        rc = lib().moe_layout_create(int(s), int(e), int(k), ctypes.byref(opt), _stream(dev), ctypes.byref(raw))
    _check(rc, "moe_layout_create")
    return Handle(raw, dev)


def moe_layout_rebuild(h: Handle, topk_idx: torch.Tensor) -> Handle:
    """Rebuild h's layout in place from new expert ids i32 [s, k]."""
    if topk_idx.dtype != torch.int32 or tuple(topk_idx.shape) != (h.s, h.k):
        raise MoEError(1, "moe_layout_rebuild", "topk_idx must be int32 [s, k] of the handle's shape")
    _check(lib().moe_layout_rebuild(h.raw, _ptr(topk_idx), _stream(topk_idx.device)), "moe_layout_rebuild")
    return h


def moe_topk_gate_layout(h: Handle, logits: torch.Tensor, renorm: int = 1, topk_idx: torch.Tensor | None = None,
                         topk_gate: torch.Tensor | None = None):
    """The top-k gate and the layout build in one kernel: logits f32 [s, e]
    -> (topk_idx i32 [s, k], topk_gate f32 [s, k]), h rebuilt on those ids."""
    if logits.dtype != torch.float32 or tuple(logits.shape) != (h.s, h.e):
        raise MoEError(1, "moe_topk_gate_layout", "logits must be float32 [s, e] of the handle's shape")
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty(h.s, h.k, dtype=torch.int32, device=dev)
    if topk_gate is None:
        topk_gate = torch.empty(h.s, h.k, dtype=torch.float32, device=dev)
    if tuple(topk_idx.shape) != (h.s, h.k) or tuple(topk_gate.shape) != (h.s, h.k) or \
            topk_idx.dtype != torch.int32 or topk_gate.dtype != torch.float32:
        raise MoEError(1, "moe_topk_gate_layout", "output shapes")
    rc = lib().moe_topk_gate_layout(h.raw, _ptr(logits), int(renorm), _ptr(topk_idx), _ptr(topk_gate), _stream(dev))
    _check(rc, "moe_topk_gate_layout")
    return topk_idx, topk_gate


def _rows2(t: torch.Tensor, name: str) -> tuple[int, int]:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    return t.shape[0], t.shape[1]


def moe_dispatch(h: Handle, x: torch.Tensor, X: torch.Tensor | None = None) -> torch.Tensor:
    """x [s,m] -> X [rows,m]."""
    s, m = _rows2(x, "x")
    if X is None:
        X = torch.empty(h.rows, m, dtype=x.dtype, device=x.device)
    rows, mX = _rows2(X, "X")
    if mX != m or X.dtype != x.dtype:
        raise MoEError(1, "moe_dispatch", "x and X disagree in width or dtype")
    _check(lib().moe_dispatch(h.raw, s, rows, m, _dtype(x), _ptr(x), _ptr(X), _stream(x.device)), "moe_dispatch")
    return X


def moe_combine(h: Handle, y: torch.Tensor, gate: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """y [rows,m], gate f32 [s,k] -> out [s,m]."""
    rows, m = _rows2(y, "y")
    if gate.dtype != torch.float32 or gate.shape != (h.s, h.k):
        raise MoEError(1, "moe_combine", "gate must be float32 [s, k]")
    if out is None:
        out = torch.empty(h.s, m, dtype=y.dtype, device=y.device)
    s, mo = _rows2(out, "out")
    if mo != m or out.dtype != y.dtype:
        raise MoEError(1, "moe_combine", "y and out disagree in width or dtype")
    _check(lib().moe_combine(h.raw, s, rows, m, _dtype(y), _ptr(y), _ptr(gate), _ptr(out), _stream(y.device)),
           "moe_combine")
    return out


def moe_combine_bwd(h: Handle, dout: torch.Tensor, gate: torch.Tensor, y: torch.Tensor,
                    dY: torch.Tensor | None = None, dgate: torch.Tensor | None = None):
    """dout [s,m], gate f32 [s,k], y [rows,m] -> (dY [rows,m], dgate f32 [s,k])."""
    s, m = _rows2(dout, "dout")
    rows, my = _rows2(y, "y")
    if my != m or y.dtype != dout.dtype:
        raise MoEError(1, "moe_combine_bwd", "dout and y disagree in width or dtype")
    if gate.dtype != torch.float32 or gate.shape != (h.s, h.k):
        raise MoEError(1, "moe_combine_bwd", "gate must be float32 [s, k]")
    if dY is None:
        dY = torch.empty(rows, m, dtype=dout.dtype, device=dout.device)
    if dgate is None:
        dgate = torch.empty(h.s, h.k, dtype=torch.float32, device=dout.device)
    if dY.shape != (rows, m) or dY.dtype != dout.dtype or dgate.shape != (h.s, h.k):
        raise MoEError(1, "moe_combine_bwd", "output shapes")
    rc = lib().moe_combine_bwd(h.raw, s, rows, m, _dtype(dout), _ptr(dout), _ptr(gate), _ptr(y), _ptr(dY),
                               _ptr(dgate), _stream(dout.device))
    _check(rc, "moe_combine_bwd")
    return dY, dgate


def moe_combine_gate_bwd(h: Handle, dout: torch.Tensor, gate: torch.Tensor, y: torch.Tensor,
                         logits: torch.Tensor | None, renorm: int = 1, dY: torch.Tensor | None = None,
                         dgate: torch.Tensor | None = None, dlogits: torch.Tensor | None = None):
    """The combine backward and the top-k gate backward in one kernel:
    (dY [rows,m], dgate f32 [s,k], dlogits f32 [s,e]); logits f32 [s,e] only
    needed when renorm = 0."""
    s, m = _rows2(dout, "dout")
    rows, my = _rows2(y, "y")
    if my != m or y.dtype != dout.dtype:
        raise MoEError(1, "moe_combine_gate_bwd", "dout and y disagree in width or dtype")
    if gate.dtype != torch.float32 or gate.shape != (h.s, h.k):
        raise MoEError(1, "moe_combine_gate_bwd", "gate must be float32 [s, k]")
    if not renorm and (logits is None or logits.dtype != torch.float32 or logits.shape != (h.s, h.e)):
        raise MoEError(1, "moe_combine_gate_bwd", "logits must be float32 [s, e] when renorm = 0")
    if dY is None:
        dY = torch.empty(rows, m, dtype=dout.dtype, device=dout.device)
    if dgate is None:
        dgate = torch.empty(h.s, h.k, dtype=torch.float32, device=dout.device)
    if dlogits is None:
        dlogits = torch.empty(h.s, h.e, dtype=torch.float32, device=dout.device)
    if dY.shape != (rows, m) or dY.dtype != dout.dtype or dgate.shape != (h.s, h.k) or \
            dlogits.shape != (h.s, h.e) or dlogits.dtype != torch.float32:
        raise MoEError(1, "moe_combine_gate_bwd", "output shapes")
    rc = lib().moe_combine_gate_bwd(h.raw, s, rows, m, _dtype(dout), _ptr(dout), _ptr(gate), _ptr(y),
                                    _ptr(None if renorm else logits), int(renorm), _ptr(dY), _ptr(dgate),
                                    _ptr(dlogits), _stream(dout.device))
    _check(rc, "moe_combine_gate_bwd")
    return dY, dgate, dlogits


def moe_dispatch_bwd(h: Handle, dX: torch.Tensor, dx: torch.Tensor | None = None) -> torch.Tensor:
    """dX [rows,m] -> dx [s,m]."""
    rows, m = _rows2(dX, "dX")
    if dx is None:
        dx = torch.empty(h.s, m, dtype=dX.dtype, device=dX.device)
    s, mx = _rows2(dx, "dx")
    if mx != m or dx.dtype != dX.dtype:
        raise MoEError(1, "moe_dispatch_bwd", "dX and dx disagree in width or dtype")
    _check(lib().moe_dispatch_bwd(h.raw, s, rows, m, _dtype(dX), _ptr(dX), _ptr(dx), _stream(dX.device)),
           "moe_dispatch_bwd")
    return dx


# ---------------------------------------------------- expert parallelism --

def moe_ep_pack(h: Handle, gate: torch.Tensor, rows_sent: int, send_row: torch.Tensor | None = None,
                meta_idx: torch.Tensor | None = None, meta_gate: torch.Tensor | None = None):
    """The send map of a source handle (built with send slots over R ranks):
    (send_row i32 [s,R], meta_idx i32 [rows_sent,k], meta_gate f32 [rows_sent,k])."""
    dev = gate.device
    if gate.dtype != torch.float32 or tuple(gate.shape) != (h.s, h.k):
        raise MoEError(1, "moe_ep_pack", "gate must be float32 [s, k]")
    if send_row is None:
        send_row = torch.empty(h.s, h.R, dtype=torch.int32, device=dev)
    if meta_idx is None:
        meta_idx = torch.empty(rows_sent, h.k, dtype=torch.int32, device=dev)
    if meta_gate is None:
        meta_gate = torch.empty(rows_sent, h.k, dtype=torch.float32, device=dev)
    if tuple(send_row.shape) != (h.s, h.R) or tuple(meta_idx.shape) != (rows_sent, h.k) or \
            tuple(meta_gate.shape) != (rows_sent, h.k):
        raise MoEError(1, "moe_ep_pack", "output shapes")
    _check(lib().moe_ep_pack(h.raw, _ptr(gate), int(rows_sent), _ptr(send_row), _ptr(meta_idx), _ptr(meta_gate),
                             _stream(dev)), "moe_ep_pack")
    return send_row, meta_idx, meta_gate


def moe_ep_dispatch(h: Handle, send_row: torch.Tensor, rows_sent: int, x: torch.Tensor,
                    X_send: torch.Tensor | None = None) -> torch.Tensor:
    """The send buffer [rows_sent, m]: each token row once per destination rank."""
    s, m = _rows2(x, "x")
    if X_send is None:
        X_send = torch.empty(rows_sent, m, dtype=x.dtype, device=x.device)
    if tuple(X_send.shape) != (rows_sent, m) or X_send.dtype != x.dtype or s != h.s:
        raise MoEError(1, "moe_ep_dispatch", "shapes")
    _check(lib().moe_ep_dispatch(h.raw, _ptr(send_row), int(rows_sent), m, _dtype(x), _ptr(x), _ptr(X_send),
                                 _stream(x.device)), "moe_ep_dispatch")
    return X_send


def moe_ep_combine(h: Handle, send_row: torch.Tensor, rows_sent: int, P: torch.Tensor,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """out [s, m] = the returned partials P [rows_sent, m] summed over ranks in rank order."""
    rows, m = _rows2(P, "P")
    if rows != rows_sent:
        raise MoEError(1, "moe_ep_combine", "P must have rows_sent rows")
    if out is None:
        out = torch.empty(h.s, m, dtype=P.dtype, device=P.device)
    if tuple(out.shape) != (h.s, m) or out.dtype != P.dtype:
        raise MoEError(1, "moe_ep_combine", "output shape")
    _check(lib().moe_ep_combine(h.raw, _ptr(send_row), int(rows_sent), m, _dtype(P), _ptr(P), _ptr(out),
                                _stream(P.device)), "moe_ep_combine")
    return out


def moe_ep_unpack_dgate(h: Handle, send_row: torch.Tensor, rows_sent: int, dgate_back: torch.Tensor,
                        dgate: torch.Tensor | None = None) -> torch.Tensor:
    """dgate f32 [s, k] from the gate gradients returned per sent row [rows_sent, k]."""
    if tuple(dgate_back.shape) != (rows_sent, h.k) or dgate_back.dtype != torch.float32:
        raise MoEError(1, "moe_ep_unpack_dgate", "dgate_back must be float32 [rows_sent, k]")
    if dgate is None:
        dgate = torch.empty(h.s, h.k, dtype=torch.float32, device=dgate_back.device)
    _check(lib().moe_ep_unpack_dgate(h.raw, _ptr(send_row), int(rows_sent), _ptr(dgate_back), _ptr(dgate),
                                     _stream(dgate_back.device)), "moe_ep_unpack_dgate")
    return dgate


def moe_grouped_gemm(h: Handle, X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor | None = None) -> torch.Tensor:
    """X bf16 [rows,K], W bf16 [e,N,K] -> Y bf16 [rows,N] per expert segment (tensor cores)."""
    rows, K = _rows2(X, "X")
    if W.dim() != 3 or W.shape[0] != h.e or W.shape[2] != K:
        raise MoEError(1, "moe_grouped_gemm", "W must be [e, N, K]")
    if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise MoEError(3, "moe_grouped_gemm", "X and W must be bf16")
    N = W.shape[1]
    if Y is None:
        Y = torch.empty(rows, N, dtype=torch.bfloat16, device=X.device)
    _check(lib().moe_grouped_gemm(h.raw, rows, K, N, _ptr(X), _ptr(W), _ptr(Y), _stream(X.device)),
           "moe_grouped_gemm")
    return Y


def moe_dispatch_grouped_gemm(h: Handle, x: torch.Tensor, W: torch.Tensor,
                              Y: torch.Tensor | None = None) -> torch.Tensor:
    """x bf16 [s,K], W bf16 [e,N,K] -> Y bf16 [rows,N]: the grouped GEMM on the
    token rows gathered through the handle, without a dispatched buffer."""
    s, K = _rows2(x, "x")
    if W.dim() != 3 or W.shape[0] != h.e or W.shape[2] != K:
        raise MoEError(1, "moe_dispatch_grouped_gemm", "W must be [e, N, K]")
    if x.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise MoEError(3, "moe_dispatch_grouped_gemm", "x and W must be bf16")
    N = W.shape[1]
    if Y is None:
        Y = torch.empty(h.rows, N, dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_dispatch_grouped_gemm(h.raw, s, h.rows, K, N, _ptr(x), _ptr(W), _ptr(Y),
                                           _stream(x.device)), "moe_dispatch_grouped_gemm")
    return Y
