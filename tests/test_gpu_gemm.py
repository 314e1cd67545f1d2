"""The expert-grouped GEMM on the tensor cores against the oracle.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all": the dispatched buffer is grouped by expert for the grouped
GEMM, groups bounded by offsets.  Identity weights must give the dispatched
rows back bit for bit (a swizzle or descriptor slip would permute them);
random weights are compared with a float64 matmul per expert segment.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as T
from combine_moe_topk_gb300 import binding as B
from combine_moe_topk_gb300 import workloads as W
from gpu_util import bits, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _setup(s, e, k, m, seed, capacity=0, pad=128):
    idx = W.random_routes(s, e, k, seed=seed)
    if capacity:
        h = B.moe_dispatch_layout(idx.to(DEV), e, capacity)
    else:
        h = B.moe_dispatch_layout_ex(idx.to(DEV), e, 0, 0, "token", pad)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(s, m, generator=g).to(torch.bfloat16)
    X = B.moe_dispatch(h, x.to(DEV))
    L = oracle.layout(idx.numpy(), e, capacity, pad_multiple=1 if capacity else pad)
    OX = oracle.dispatch(L["row"], bits(x), L["rows"])
    np.testing.assert_array_equal(bits(X), OX)
    return h, X, OX, L


def _owned_rows(L):
    rows = []
    for x in range(len(L["counts"])):
        rows.extend(range(int(L["offsets"][x]), int(L["offsets"][x]) + int(L["counts"][x])))
    return np.array(rows, np.int64)


def test_identity_weights_return_the_dispatched_rows():
    s, e, k, K = 300, 4, 2, 256
    h, X, OX, L = _setup(s, e, k, K, seed=1)
    Wt = torch.eye(K, dtype=torch.bfloat16).expand(e, K, K).contiguous()
    Y = B.moe_grouped_gemm(h, X, Wt.to(DEV))
    torch.cuda.synchronize()
    assert h.status() == 0
    r = _owned_rows(L)
    np.testing.assert_array_equal(bits(Y)[r], OX[r])


@pytest.mark.parametrize("case", [
    dict(s=150, e=2, k=1, K=64, N=256, cap=0),
    dict(s=2000, e=8, k=2, K=1024, N=512, cap=0),
    dict(s=1500, e=6, k=3, K=512, N=768, cap=768),     # capacity mode, 128-aligned slots
    dict(s=4096, e=16, k=4, K=2048, N=256, cap=0),
])
def test_grouped_gemm_matches_float64_matmul(case):
    s, e, k, K, N, cap = case["s"], case["e"], case["k"], case["K"], case["N"], case["cap"]
    h, X, OX, L = _setup(s, e, k, K, seed=3, capacity=cap)
    g = torch.Generator().manual_seed(7)
    Wt = (torch.randn(e, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    Y = B.moe_grouped_gemm(h, X, Wt.to(DEV))
    torch.cuda.synchronize()
    assert h.status() == 0
    Wb = bits(Wt)
    ref = oracle.grouped_gemm(OX, Wb, L["offsets"], L["counts"])
    r = _owned_rows(L)
    got = T.as_f64(bits(Y)[r])
    # bf16 output: one ulp of the exact value plus the fp32 accumulation over K
    scale = np.zeros_like(ref[r])
    Xa, Wa = np.abs(T.as_f64(OX)), np.abs(T.as_f64(Wb))
    for x in range(e):
        o, n = int(L["offsets"][x]), int(L["counts"][x])
        sel = (r >= o) & (r < o + n)
        scale[sel] = Xa[r[sel]] @ Wa[x].T
    bad = np.abs(got - ref[r]) > T.bf16_ulp(ref[r]) + 1e-5 * scale
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3])


def test_unaligned_segments_are_refused():
    idx = W.random_routes(100, 4, 2, seed=2).to(DEV)
    h = B.moe_dispatch_layout_ex(idx, 4, 0, 0, "token", 4)
    X = torch.zeros(h.rows, 64, dtype=torch.bfloat16, device=DEV)
    Wt = torch.zeros(4, 256, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(B.MoEError) as ei:
        B.moe_grouped_gemm(h, X, Wt)
    assert ei.value.name == "MOE_ERR_UNSUPPORTED"
