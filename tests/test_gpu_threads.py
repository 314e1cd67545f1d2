"""The library called from several host threads at once.

ctypes releases the GIL around foreign calls, so the C entry points really
run concurrently here: the handle registry, the once-per-device set-up and
the per-thread error string are shared state.  Each thread builds layouts
and runs dispatch / combine / backward on its own stream and inputs; every
result must equal the same computation done single-threaded beforehand.
"""
import threading

import pytest
import torch

from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(inp, w, stream):
    with torch.cuda.stream(stream):
        idx, gate = B.moe_topk_gate(inp["logits"], w.k, w.renorm)
        h = B.moe_dispatch_layout(idx, w.e, w.capacity, w.R)
        X = B.moe_dispatch(h, inp["x"])
        out = B.moe_combine(h, inp["y"], gate)
        dY, dgate = B.moe_combine_bwd(h, inp["dout"], gate, inp["y"])
        dx = B.moe_dispatch_bwd(h, dY)
        stream.synchronize()
        status = h.status()
        res = [t.clone() for t in (idx, gate, h.row(), X, out, dY, dgate, dx)]
        h.destroy()
    return status, res


def test_concurrent_host_threads_match_serial_results():
    w = W.WORKLOADS["fine-grained-skewed"].replace(s=1500, m=256)
    inputs = [W.make_inputs(w, device=DEV, seed=100 + i) for i in range(4)]
    serial = [_run(inp, w, torch.cuda.Stream(DEV))[1] for inp in inputs]
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream(DEV)
            for _ in range(15):
                status, res = _run(inputs[i], w, stream)
                assert status == 0
                for a, b in zip(res, serial[i]):
                    assert torch.equal(a, b)
            # a rejected call's message stays with the thread that made it
            with pytest.raises(B.MoEError):
                B.moe_dispatch_layout(torch.zeros(4, 2, dtype=torch.int32, device=DEV), 6, 0, 4)  # R must divide e
        except Exception as exc:  # surfaced to the main thread below
            errors.append((i, repr(exc)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
