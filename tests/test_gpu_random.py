"""The whole path on the GPU against the oracle over seeded random shapes.

Each case draws a workload (tokens, width, experts, k, activation type,
capacity or dropless, capacity priority, per-expert padding, virtual ranks,
expert skew, gate renormalisation) from a fixed seed and runs gate, layout,
dispatch, combine and both backwards on the GPU and in the oracle on the
same inputs: indices, layouts and dispatched rows bit-exact, gates and the
fp32-accumulated results within the stated tolerances.  The draws reach
shapes the named workloads do not: widths of a few 16-byte vectors, one or
three experts, k = e, a capacity of one slot, pads larger than most
segments, odd token counts.
"""
import numpy as np
import pytest

from combine_moe_topk_gb300 import workloads as W
from gpu_util import full_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def draw_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        e = int(rng.choice([1, 2, 3, 5, 8, 12, 16, 64, 128, 256]))
        k = int(rng.integers(1, min(e, 16) + 1))
        s = int(rng.integers(1, 3000))
        dtype = str(rng.choice(["f32", "bf16"]))
        m = int(rng.integers(1, 48)) * (4 if dtype == "f32" else 8)
        capacity = 0 if rng.random() < 0.5 else int(rng.integers(1, max(2, 2 * s * k // e)))
        priority = "kmajor" if rng.random() < 0.3 else "token"
        pad = 1 if capacity or rng.random() < 0.6 else int(rng.choice([2, 8, 64, 128]))
        divisors = [r for r in range(1, min(e, 64) + 1) if e % r == 0]
        R = 0 if rng.random() < 0.4 else int(rng.choice(divisors))
        zipf = float(rng.choice([0.0, 0.0, 1.2, 3.0]))
        renorm = int(rng.integers(0, 2))
        w = W.Workload(f"random{i}", s=s, m=m, e=e, k=k, dtype=dtype, capacity=capacity, R=R,
                       seed=int(rng.integers(0, 2**31 - 1)), zipf_alpha=zipf, renorm=renorm)
        cases.append((w, priority, pad))
    return cases


CASES = draw_cases(48, seed=20261202)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-s{c[0].s}-m{c[0].m}-e{c[0].e}-k{c[0].k}-"
                                                      f"{c[0].dtype}-c{c[0].capacity}-{c[1]}-p{c[2]}-R{c[0].R}")
def test_random_shapes_match_the_oracle(case):
    w, priority, pad = case
    full_parity(w, DEV, priority=priority, pad_multiple=pad)
