"""Autograd wrappers and the activation-checkpoint handle recorder.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all", description: the backward of a combine is a dispatch and the
backward of a dispatch is a combine, both replayed against the handle the
forward layout produced; review thread: the routing weights are an autograd
input of the combine, so their gradient reaches the router.

Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
activation-checkpoint recompute", "How": one recorder per checkpointed call;
the forward logs each dispatch's handle and routing metadata in call order,
the recompute consumes them in the same order, the dispatched activation is
not retained, and a replay that outruns its log falls back to a full layout
build rather than replaying a mismatched one.  Replay is only valid when the
routing is pinned across recompute; the recorder checks the expert ids it is
given against the logged ones (on the device) when asked to.

All arithmetic runs in the CUDA library (``binding``); this module only
wires tensors and handles together.
"""
from __future__ import annotations

from collections import deque

import torch

from . import binding as B


class MoETopkGateFn(torch.autograd.Function):
    """(idx, gate) = topk_gate(logits); dlogits = topk_gate_bwd(dgate).  The
    expert ids are not differentiable; the gates' gradient reaches the router."""

    @staticmethod
    def forward(ctx, logits: torch.Tensor, k: int, renorm: int):
        logits = logits.contiguous()
        idx, gate = B.moe_topk_gate(logits, k, renorm)
        ctx.renorm = int(renorm)
        ctx.e = logits.shape[1]
        ctx.save_for_backward(None if renorm else logits, idx, gate)
        ctx.mark_non_differentiable(idx)
        return idx, gate

    @staticmethod
    def backward(ctx, didx, dgate: torch.Tensor):
        logits, idx, gate = ctx.saved_tensors
        dl = B.moe_topk_gate_bwd(logits, idx, gate, dgate.contiguous(), ctx.e, ctx.renorm)
        return dl, None, None


def topk_gate(logits: torch.Tensor, k: int, renorm: int = 1):
    return MoETopkGateFn.apply(logits, k, renorm)


class MoEDispatchFn(torch.autograd.Function):
    """X = dispatch(x) on a layout handle; dx = dispatch_bwd(dX) on the same handle."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, handle: B.Handle):
        ctx.handle = handle
        return B.moe_dispatch(handle, x.contiguous())

    @staticmethod
    def backward(ctx, dX: torch.Tensor):
        return B.moe_dispatch_bwd(ctx.handle, dX.contiguous()), None


class MoECombineFn(torch.autograd.Function):
    """out = combine(y, gate); (dY, dgate) = combine_bwd(dout, gate, y)."""

    @staticmethod
    def forward(ctx, y: torch.Tensor, gate: torch.Tensor, handle: B.Handle):
        y = y.contiguous()
        gate = gate.contiguous()
        ctx.handle = handle
        ctx.save_for_backward(y, gate)
        return B.moe_combine(handle, y, gate)

    @staticmethod
    def backward(ctx, dout: torch.Tensor):
        y, gate = ctx.saved_tensors
        dY, dgate = B.moe_combine_bwd(ctx.handle, dout.contiguous(), gate, y)
        return dY, dgate, None


def dispatch(x: torch.Tensor, handle: B.Handle) -> torch.Tensor:
    return MoEDispatchFn.apply(x, handle)


def combine(y: torch.Tensor, gate: torch.Tensor, handle: B.Handle) -> torch.Tensor:
    return MoECombineFn.apply(y, gate, handle)


class HandleRecorder:
    """Per-checkpointed-call log of layout handles.

    ``layout(topk_idx, ...)`` builds a fresh layout while recording (the
    forward) and appends it to the log; once ``replay()`` is entered (the
    recompute) it returns the logged handles in call order without
    launching the layout kernel.  A replay past the end of the log builds a
    fresh layout (``fallbacks`` counts those).  ``build`` is the layout
    constructor, injectable so the bookkeeping can be tested without a GPU.
    """

    def __init__(self, build=None, verify: bool = False):
        self._build = build or _build_layout
        self._log: deque = deque()
        self._replaying = False
        self.verify = verify
        self.recorded = 0
        self.replayed = 0
        self.fallbacks = 0

    def replay(self):
        """Switch to replay mode (the recompute of the checkpointed call)."""
        self._replaying = True
        return self

    def record(self):
        self._replaying = False
        self._log.clear()
        return self

    def __len__(self):
        return len(self._log)

    def layout(self, topk_idx: torch.Tensor, e: int, capacity: int = 0, num_virtual_ranks: int = 0,
               priority: str = "token", pad_multiple: int = 1, send_slots: bool = False):
        """The layout of ``topk_idx`` (options as ``moe_dispatch_layout_ex``):
        built and logged while recording, the logged handle while replaying."""
        opts = {}
        if priority != "token" or pad_multiple != 1 or send_slots:
            opts = dict(priority=priority, pad_multiple=int(pad_multiple), send_slots=bool(send_slots))
        key = (tuple(topk_idx.shape), int(e), int(capacity), int(num_virtual_ranks), tuple(sorted(opts.items())))
        if not self._replaying:
            h = self._build(topk_idx, e, capacity, num_virtual_ranks, **opts)
            # routing metadata: the expert ids; the dispatched activation is not kept
            self._log.append((key, h, topk_idx.detach() if self.verify else None))
            self.recorded += 1
            return h
        if self._log:
            k0, h, logged_idx = self._log.popleft()
            if k0 == key and (logged_idx is None or torch.equal(logged_idx, topk_idx)):
                self.replayed += 1
                return h
        # outran the log, or the call does not match what was logged: build afresh
        self.fallbacks += 1
        return self._build(topk_idx, e, capacity, num_virtual_ranks, **opts)


def _build_layout(topk_idx, e, capacity, num_virtual_ranks, priority="token", pad_multiple=1, send_slots=False):
    """Plain layouts through moe_dispatch_layout, variants through _ex."""
    if priority == "token" and pad_multiple == 1 and not send_slots:
        return B.moe_dispatch_layout(topk_idx, e, capacity, num_virtual_ranks)
    return B.moe_dispatch_layout_ex(topk_idx, e, capacity, num_virtual_ranks, priority, pad_multiple, send_slots)
