"""The allocation-free layout entry point, against the handle-building one.

``moe_dispatch_layout_noalloc`` exists for callers that cannot allocate
device memory when they build a layout -- code inside a captured CUDA graph
that must not add pool allocations, an allocator's own hook that must not
re-enter it, runtimes that only hand out fixed buffers.  It writes the same
layout into arrays the caller owns, with its scratch in a fixed library
array.  This file runs last so that a failure here leaves every other test
already run; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def layout_noalloc(idx, e, capacity, R):
    """Call the C entry point directly; outputs allocated here by the test."""
    s, k = idx.shape
    i32 = dict(dtype=torch.int32, device=DEV)
    out = {
        "idx": torch.empty(s, k, **i32), "loc": torch.empty(s, k, **i32), "row": torch.empty(s, k, **i32),
        "drop": torch.empty(s, k, dtype=torch.uint8, device=DEV),
        "raw_counts": torch.empty(e, **i32), "counts": torch.empty(e, **i32), "offsets": torch.empty(e + 1, **i32),
        "token_in_rank": torch.empty(s, R, dtype=torch.uint8, device=DEV) if R else None,
        "rank_counts": torch.full((R,), 12345, **i32) if R else None,  # must be cleared by the call
        "status": torch.zeros(1, **i32),
    }
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    rc = B.lib().moe_dispatch_layout_noalloc(
        _p(idx), s, e, k, capacity, R, _p(out["idx"]), _p(out["loc"]), _p(out["row"]), _p(out["drop"]),
        _p(out["raw_counts"]), _p(out["counts"]), _p(out["offsets"]), _p(out["token_in_rank"]),
        _p(out["rank_counts"]), _p(out["status"]), stream)
    assert rc == 0, f"{B.STATUS[rc]}: {B.lib().moe_last_error().decode()}"
    return out


def assert_same_layout(got, h):
    """Integer outputs: bit-exact, the bar every layout test uses."""
    ref = {"idx": h.idx(), "loc": h.loc(), "row": h.row(), "drop": h.drop(), "raw_counts": h.raw_counts(),
           "counts": h.counts(), "offsets": h.offsets()}
    if h.R:
        ref["token_in_rank"] = h.token_in_rank()
        ref["rank_counts"] = h.rank_counts()
    for name, want in ref.items():
        assert torch.equal(got[name], want), name
    assert int(got["status"].item()) == 0


CASES = [
    W.WORKLOADS["fine-grained-skewed"],                                  # dropless, dedup over 8 ranks
    W.WORKLOADS["gshard-capacity"],                                      # capacity 3072 with drops
    W.WORKLOADS["fine-grained-skewed"].replace(s=3001, zipf_alpha=0.0),  # smaller, after a larger call
]


def assert_oracle_layout(got, idx, e, capacity, R):
    """The same arrays against the CPU oracle's layout of the same routes."""
    ids = idx.cpu().numpy()
    L = oracle.layout(ids, e, capacity, R)
    np.testing.assert_array_equal(got["idx"].cpu().numpy(), ids, err_msg="idx")
    for name in ("loc", "row", "drop", "raw_counts", "counts", "offsets") + (("token_in_rank", "rank_counts")
                                                                              if R else ()):
        np.testing.assert_array_equal(got[name].cpu().numpy(), L[name], err_msg=name)


def test_noalloc_layout_matches_handle_layout_on_consecutive_calls():
    for w in CASES:
        logits = W.make_logits(w, device=DEV)
        idx, _ = B.moe_topk_gate(logits, w.k, w.renorm)
        h = B.moe_dispatch_layout(idx, w.e, w.capacity, w.R)
        got = layout_noalloc(idx, w.e, w.capacity, w.R)
        torch.cuda.synchronize()
        assert_same_layout(got, h)
        assert_oracle_layout(got, idx, w.e, w.capacity, w.R)
        assert h.status() == 0
        h.destroy()


def test_noalloc_largest_plan_fits_its_scratch():
    """256 experts over many tokens: the tile plan uses the whole fixed
    scratch (tiles x e = 16384 words) and still matches the handle path."""
    s, e, k = 1 << 17, 256, 4
    idx = W.random_routes(s, e, k, device=DEV, seed=3)
    h = B.moe_dispatch_layout(idx, e, 0, 8)
    got = layout_noalloc(idx, e, 0, 8)
    torch.cuda.synchronize()
    assert_same_layout(got, h)
