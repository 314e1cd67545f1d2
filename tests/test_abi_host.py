"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point the header declares, the host-only helpers
compute what they say, and invalid arguments are rejected before anything
touches CUDA.  Also the activation-checkpoint recorder's bookkeeping, with
fake handles."""
import ctypes
import os
import re

import pytest

from combine_moe_topk_gb300 import autograd as A
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import build as cuda_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_are_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    assert sorted(B.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_capacity_formula(lib):
    # ceil(cf * s * k / e): the two capacity workloads, and edge cases
    assert B.moe_capacity(1.25, 256, 2, 8) == 80
    assert B.moe_capacity(1.0, 32768, 6, 64) == 3072
    assert B.moe_capacity(1.0, 5000, 6, 64) == 469
    assert B.moe_capacity(1.0, 1, 1, 8) == 1
    assert B.moe_capacity(2.0, 0, 2, 8) == 0
    assert B.moe_capacity(0.0, 10, 2, 8) == 0
    assert B.moe_capacity(-1.0, 10, 2, 8) == 0
    assert B.moe_capacity(1.0, 10, 0, 8) == 0


def test_status_strings(lib):
    for code, name in B.STATUS.items():
        assert isinstance(B.moe_status_string(code), str) and B.moe_status_string(code)
    assert "fp32" in B.moe_status_string(3)


P = ctypes.c_void_p


def rc_name(rc):
    return B.STATUS[rc]


def test_gate_rejects_bad_sizes_without_a_gpu(lib):
    fake = P(0x10000)
    assert rc_name(lib.moe_topk_gate(fake, 4, 8, 9, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # k > e
    assert rc_name(lib.moe_topk_gate(fake, 4, 0, 1, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # e = 0
    assert rc_name(lib.moe_topk_gate(fake, 4, 300, 2, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # e > 256
    assert rc_name(lib.moe_topk_gate(fake, 4, 32, 17, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # k > 16
    assert rc_name(lib.moe_topk_gate(fake, 4, 8, 2, 2, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # renorm
    assert rc_name(lib.moe_topk_gate(None, 4, 8, 2, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # NULL
    assert rc_name(lib.moe_topk_gate(P(0x10004), 4, 8, 2, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"  # align
    assert rc_name(lib.moe_topk_gate(fake, -1, 8, 2, 1, fake, fake, None, None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_topk_gate(fake, 0, 8, 2, 1, fake, fake, None, None)) == "MOE_OK"  # empty: nothing to do
    assert "min(e, 16)" in lib.moe_last_error().decode()


def test_layout_rejects_bad_sizes_without_a_gpu(lib):
    fake = P(0x10000)
    out = P()
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 8, 2, 0, 3, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"  # R | e
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 8, 2, -1, 0, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 256, 2, 0, 128, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 8, 9, 0, 0, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_layout(fake, 2**30, 8, 4, 0, 0, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 8, 2, 2**29, 0, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_layout(fake, 4, 8, 2, 0, 0, None, None)) == "MOE_ERR_INVALID_ARG"
    assert out.value is None
    # send slots need virtual ranks; the flag is 0 or 1
    opt = B.LayoutOptions(0, 0, 0, 1, 1)
    assert rc_name(lib.moe_dispatch_layout_ex(fake, 4, 8, 2, ctypes.byref(opt), None, ctypes.byref(out))) \
        == "MOE_ERR_INVALID_ARG"
    assert "num_virtual_ranks" in lib.moe_last_error().decode()
    opt = B.LayoutOptions(0, 2, 0, 1, 2)
    assert rc_name(lib.moe_dispatch_layout_ex(fake, 4, 8, 2, ctypes.byref(opt), None, ctypes.byref(out))) \
        == "MOE_ERR_INVALID_ARG"
    assert out.value is None
    # an empty handle for in-place builds: the same checks, before any CUDA call
    assert rc_name(lib.moe_layout_create(4, 8, 2, ctypes.byref(B.LayoutOptions(0, 3, 0, 1, 0)), None,
                                         ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_layout_create(4, 8, 9, ctypes.byref(B.LayoutOptions(0, 0, 0, 1, 0)), None,
                                         ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_layout_create(4, 8, 2, None, None, ctypes.byref(out))) == "MOE_ERR_INVALID_ARG"
    assert out.value is None


def test_unknown_handles_are_rejected_without_a_gpu(lib):
    bogus = P(0xdead0)
    fake = P(0x10000)
    assert rc_name(lib.moe_dispatch(None, 4, 8, 8, 0, fake, fake, None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch(bogus, 4, 8, 8, 0, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_combine(bogus, 4, 8, 8, 1, fake, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_combine_bwd(bogus, 4, 8, 8, 1, fake, fake, fake, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_dispatch_bwd(bogus, 4, 8, 8, 1, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_combine_gate_bwd(bogus, 4, 8, 8, 1, fake, fake, fake, None, 1, fake, fake, fake,
                                            None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_combine_gate_bwd(None, 4, 8, 8, 1, fake, fake, fake, None, 1, fake, fake, fake,
                                            None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_layout_rebuild(bogus, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_layout_rebuild(None, fake, None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_topk_gate_layout(bogus, fake, 1, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_grouped_gemm(None, 8, 64, 64, fake, fake, fake, None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_grouped_gemm(bogus, 8, 64, 64, fake, fake, fake, None)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_dispatch_grouped_gemm(None, 4, 8, 64, 64, fake, fake, fake, None)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_dispatch_grouped_gemm(bogus, 4, 8, 64, 64, fake, fake, fake, None)) \
        == "MOE_ERR_HANDLE_MISMATCH"
    info = B.LayoutInfo()
    assert rc_name(lib.moe_handle_info(bogus, ctypes.byref(info))) == "MOE_ERR_HANDLE_MISMATCH"
    st = ctypes.c_int32()
    assert rc_name(lib.moe_handle_status(bogus, None, ctypes.byref(st))) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_handle_destroy(bogus)) == "MOE_ERR_HANDLE_MISMATCH"
    assert rc_name(lib.moe_handle_destroy(None)) == "MOE_ERR_INVALID_ARG"


def test_debug_hook_arguments(lib):
    assert rc_name(lib.moe_debug_hold_layout_tile(1, 0)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_debug_hold_layout_tile(1, 20000)) == "MOE_ERR_INVALID_ARG"
    assert rc_name(lib.moe_debug_hold_layout_tile(-1, 100)) == "MOE_OK"


def test_launch_counters_exist(lib):
    for name in B.KERNELS:
        assert B.moe_launch_count(name) >= 0
    assert lib.moe_launch_count(99) == 0


# ------------------------------------------------------------- recorder --

class FakeIdx:
    def __init__(self, shape, tag):
        self.shape = shape
        self.tag = tag

    def detach(self):
        return self


def test_recorder_replays_in_call_order_and_falls_back():
    built = []

    def build(idx, e, cap, R):
        h = ("handle", len(built), idx.tag)
        built.append(h)
        return h

    rec = A.HandleRecorder(build=build)
    a, b, c = FakeIdx((8, 2), "a"), FakeIdx((8, 2), "b"), FakeIdx((8, 2), "c")
    fwd = [rec.layout(a, 4), rec.layout(b, 4), rec.layout(c, 4)]
    assert rec.recorded == 3 and len(built) == 3
    rec.replay()
    assert [rec.layout(a, 4), rec.layout(b, 4), rec.layout(c, 4)] == fwd
    assert rec.replayed == 3 and len(built) == 3, "replay must not build layouts"
    extra = rec.layout(a, 4)  # outran the log: a fresh build, not a stale handle
    assert rec.fallbacks == 1 and extra == built[-1] and len(built) == 4


def test_recorder_refuses_a_mismatched_call():
    built = []

    def build(idx, e, cap, R):
        built.append(idx.tag)
        return idx.tag

    rec = A.HandleRecorder(build=build)
    rec.layout(FakeIdx((8, 2), "a"), 4, capacity=3)
    rec.replay()
    # same call position, but a different capacity: never replay a mismatched layout
    assert rec.layout(FakeIdx((8, 2), "z"), 4, capacity=5) == "z"
    assert rec.fallbacks == 1 and rec.replayed == 0


def test_per_call_recorders_keep_passes_apart():
    """One recorder per checkpointed call: three passes through the same block
    route differently and must each replay their own handles."""
    built = []

    def build(idx, e, cap, R):
        built.append(idx.tag)
        return idx.tag

    recs = [A.HandleRecorder(build=build) for _ in range(3)]
    for p, rec in enumerate(recs):
        for layer in range(4):
            rec.layout(FakeIdx((8, 2), f"p{p}l{layer}"), 4)
    n = len(built)
    for p in (2, 0):  # recompute order: later passes first
        recs[p].replay()
        assert [recs[p].layout(FakeIdx((8, 2), "?"), 4) for _ in range(4)] == [f"p{p}l{l}" for l in range(4)]
    assert len(built) == n


def test_recorder_keys_on_layout_options():
    """A replay must match the logged call's layout options too: k-major,
    padding and send slots are part of what was built."""
    built = []

    def build(idx, e, cap, R, **opts):
        built.append((idx.tag, opts))
        return idx.tag

    rec = A.HandleRecorder(build=build)
    rec.layout(FakeIdx((8, 2), "a"), 4, capacity=3, priority="kmajor")
    rec.layout(FakeIdx((8, 2), "b"), 4, pad_multiple=8, send_slots=False)
    assert built[0][1] == {"priority": "kmajor", "pad_multiple": 1, "send_slots": False}
    rec.replay()
    assert rec.layout(FakeIdx((8, 2), "?"), 4, capacity=3, priority="kmajor") == "a"
    # same call position, but token priority this time: rebuilt, not replayed
    assert rec.layout(FakeIdx((8, 2), "c"), 4, pad_multiple=1) == "c"
    assert rec.replayed == 1 and rec.fallbacks == 1
