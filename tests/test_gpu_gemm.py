"""The expert-grouped GEMM on the tensor cores, plain and fused with the
dispatch, against the oracle.

DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
all-to-all": the dispatched buffer is grouped by expert for the grouped
GEMM, groups bounded by offsets.  Identity weights must give the dispatched
rows back bit for bit (a swizzle, descriptor or gather slip would permute
them); random weights are compared with a float64 matmul per expert segment.
The fused form gathers the token rows itself and must equal the plain GEMM
on the dispatched rows bit for bit (same operands, same MMA order).  Rows no
route owns are left as they were.
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
SENTINEL = 0x7FC1  # a bf16 NaN pattern no GEMM result equals


def _setup(s, e, k, m, seed, capacity=0, pad=1, priority="token"):
    idx = W.random_routes(s, e, k, seed=seed)
    if pad > 1 or priority != "token":
        h = B.moe_dispatch_layout_ex(idx.to(DEV), e, capacity, 0, priority, pad)
    else:
        h = B.moe_dispatch_layout(idx.to(DEV), e, capacity)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(s, m, generator=g).to(torch.bfloat16)
    X = B.moe_dispatch(h, x.to(DEV))
    L = oracle.layout(idx.numpy(), e, capacity, priority=1 if priority == "kmajor" else 0,
                      pad_multiple=pad)
    OX = oracle.dispatch(L["row"], bits(x), L["rows"])
    np.testing.assert_array_equal(bits(X), OX)
    return h, x, X, OX, L


def _owned_rows(L):
    rows = []
    for x in range(len(L["counts"])):
        rows.extend(range(int(L["offsets"][x]), int(L["offsets"][x]) + int(L["counts"][x])))
    return np.array(rows, np.int64)


def _sentinel_out(rows, N):
    return torch.full((rows, N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)


def _check_unowned_untouched(Y, L):
    own = np.zeros(int(L["rows"]), bool)
    own[_owned_rows(L)] = True
    rest = bits(Y)[~own]
    assert (rest == SENTINEL).all(), "a row no route owns was written"


def _check_float64(Y, OX, Wt, L):
    Wb = bits(Wt)
    ref = oracle.grouped_gemm(OX, Wb, L["offsets"], L["counts"])
    r = _owned_rows(L)
    got = T.as_f64(bits(Y)[r])
    # bf16 output: one ulp of the exact value plus the fp32 accumulation over K
    scale = np.zeros_like(ref[r])
    Xa, Wa = np.abs(T.as_f64(OX)), np.abs(T.as_f64(Wb))
    for x in range(len(L["counts"])):
        o, n = int(L["offsets"][x]), int(L["counts"][x])
        sel = (r >= o) & (r < o + n)
        scale[sel] = Xa[r[sel]] @ Wa[x].T
    bad = np.abs(got - ref[r]) > T.bf16_ulp(ref[r]) + 1e-5 * scale
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3])


@pytest.mark.parametrize("K", [256, 72])  # 72: a K tail and a partial column tile
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("layout", [dict(pad=128), dict(pad=1), dict(capacity=100)])
def test_identity_weights_return_the_dispatched_rows(fused, layout, K):
    s, e, k = 300, 4, 2
    h, x, X, OX, L = _setup(s, e, k, K, seed=1, **layout)
    Wt = torch.eye(K, dtype=torch.bfloat16).expand(e, K, K).contiguous().to(DEV)
    Y = _sentinel_out(h.rows, K)
    if fused:
        B.moe_dispatch_grouped_gemm(h, x.to(DEV), Wt, Y)
    else:
        B.moe_grouped_gemm(h, X, Wt, Y)
    torch.cuda.synchronize()
    assert h.status() == 0
    r = _owned_rows(L)
    np.testing.assert_array_equal(bits(Y)[r], OX[r])
    _check_unowned_untouched(Y, L)


CASES = [
    dict(s=150, e=2, k=1, K=64, N=256),
    dict(s=2000, e=8, k=2, K=1024, N=512),                       # plain dropless: segments start anywhere
    dict(s=1500, e=6, k=3, K=512, N=768, capacity=768),          # capacity, 128-aligned slots
    dict(s=1500, e=6, k=3, K=512, N=256, capacity=333),          # capacity, unaligned slots, drops
    dict(s=4096, e=16, k=4, K=2048, N=256, pad=128),             # padded
    dict(s=3000, e=64, k=6, K=256, N=512, capacity=200, priority="kmajor"),
    dict(s=700, e=128, k=8, K=128, N=256),                       # many small and empty segments
    dict(s=40, e=4, k=1, K=64, N=256),                           # fewer rows than one block
    dict(s=900, e=256, k=4, K=64, N=256),                        # the largest expert count
    dict(s=1200, e=8, k=2, K=72, N=264),                         # K and N tails: K % 64, N % 256 != 0
    dict(s=700, e=6, k=2, K=1000, N=1416, capacity=250),         # tails in capacity mode
    dict(s=500, e=4, k=2, K=64, N=8),                            # one 8-column chunk
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_grouped_gemm_matches_float64_matmul_and_fused_is_identical(case):
    c = dict(case)
    s, e, k, K, N = (c.pop(n) for n in ("s", "e", "k", "K", "N"))
    h, x, X, OX, L = _setup(s, e, k, K, seed=3, **c)
    g = torch.Generator().manual_seed(7)
    Wt = (torch.randn(e, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    Wd = Wt.to(DEV)
    Y = B.moe_grouped_gemm(h, X, Wd, _sentinel_out(h.rows, N))
    Yf = B.moe_dispatch_grouped_gemm(h, x.to(DEV), Wd, _sentinel_out(h.rows, N))
    torch.cuda.synchronize()
    assert h.status() == 0
    _check_float64(Y, OX, Wt, L)
    np.testing.assert_array_equal(bits(Yf), bits(Y))  # owned rows equal, the rest untouched in both
    _check_unowned_untouched(Y, L)


SEGMENT_COUNTS = [0, 1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 640]


@pytest.mark.parametrize("weights", ["identity", "random"])
def test_segments_around_the_block_edges(weights):
    """Expert segments of every size class at the 128- and 256-row block
    edges of the pair kernel's 256-row blocks (each CTA's 128-row half):
    empty, full blocks only (256), a last block whose second half holds
    1..127 rows (129, 255, 257 .. 511) or none (1, 127, 128, 384, 640);
    plain and fused, every owned row against the oracle, the rest untouched."""
    e = len(SEGMENT_COUNTS)
    ids = np.repeat(np.arange(e), SEGMENT_COUNTS)
    rng = np.random.default_rng(17)
    rng.shuffle(ids)  # token order across experts
    s, K = len(ids), 128
    idx = torch.from_numpy(ids.astype(np.int32)).view(s, 1)
    h = B.moe_dispatch_layout(idx.to(DEV), e)
    L = oracle.layout(idx.numpy(), e)
    np.testing.assert_array_equal(np.asarray(L["counts"]), SEGMENT_COUNTS)
    g = torch.Generator().manual_seed(19)
    x = torch.randn(s, K, generator=g).to(torch.bfloat16)
    X = B.moe_dispatch(h, x.to(DEV))
    OX = oracle.dispatch(L["row"], bits(x), L["rows"])
    if weights == "identity":
        N = K
        Wt = torch.eye(K, dtype=torch.bfloat16).expand(e, K, K).contiguous()
    else:
        N = 264  # a partial second column tile
        Wt = (torch.randn(e, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    Wd = Wt.to(DEV)
    Y = B.moe_grouped_gemm(h, X, Wd, _sentinel_out(h.rows, N))
    Yf = B.moe_dispatch_grouped_gemm(h, x.to(DEV), Wd, _sentinel_out(h.rows, N))
    torch.cuda.synchronize()
    assert h.status() == 0
    if weights == "identity":
        r = _owned_rows(L)
        np.testing.assert_array_equal(bits(Y)[r], OX[r])
    else:
        _check_float64(Y, OX, Wt, L)
    np.testing.assert_array_equal(bits(Yf), bits(Y))
    _check_unowned_untouched(Y, L)


def test_inv_row_names_the_token_of_every_owned_row():
    s, e, k = 5000, 32, 4
    for kw in (dict(capacity=500), dict(capacity=0), dict(capacity=600, priority="kmajor")):
        idx = W.random_routes(s, e, k, seed=9)
        pri = kw.get("priority", "token")
        h = B.moe_dispatch_layout_ex(idx.to(DEV), e, kw["capacity"], 0, pri, 1)
        L = oracle.layout(idx.numpy(), e, kw["capacity"], priority=1 if pri == "kmajor" else 0)
        want = np.full(int(L["rows"]), -1, np.int64)
        t, j = np.nonzero(L["row"] >= 0)
        want[L["row"][t, j]] = t
        r = _owned_rows(L)
        np.testing.assert_array_equal(bits(h.inv_row())[r], want[r])


def test_gemm_argument_checks():
    idx = W.random_routes(100, 4, 2, seed=2).to(DEV)
    h = B.moe_dispatch_layout(idx, 4)
    bf = dict(dtype=torch.bfloat16, device=DEV)
    with pytest.raises(B.MoEError) as ei:
        B.moe_grouped_gemm(h, torch.zeros(h.rows, 100, **bf), torch.zeros(4, 256, 100, **bf))
    assert ei.value.name == "MOE_ERR_INVALID_ARG"  # K = 100: not a multiple of 8
    with pytest.raises(B.MoEError) as ei:
        B.moe_grouped_gemm(h, torch.zeros(h.rows, 56, **bf), torch.zeros(4, 256, 56, **bf))
    assert ei.value.name == "MOE_ERR_INVALID_ARG"  # K = 56 < 64
    x = torch.zeros(101, 64, **bf)
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch_grouped_gemm(h, x, torch.zeros(4, 256, 64, **bf))
    assert ei.value.name == "MOE_ERR_HANDLE_MISMATCH"  # 101 token rows, the handle has 100
    with pytest.raises(B.MoEError) as ei:
        B.moe_grouped_gemm(h, torch.zeros(h.rows, 64, **bf), torch.zeros(4, 200 + 4, 64, **bf))
    assert ei.value.name == "MOE_ERR_INVALID_ARG"  # N = 204: not a multiple of 8


def test_fused_pair_is_stable_over_repeated_calls():
    """The fused form's second CTA signals its gathered rows through a
    shared-to-shared bulk copy; any ordering slip would show as rows that
    differ from call to call.  40 calls, each compared bit for bit with the
    plain GEMM on the dispatched rows."""
    s, e, k, K, N = 3000, 16, 4, 512, 512
    h, x, X, OX, L = _setup(s, e, k, K, seed=11)
    g = torch.Generator().manual_seed(13)
    Wd = (torch.randn(e, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16).to(DEV)
    ref = B.moe_grouped_gemm(h, X, Wd)
    xd = x.to(DEV)
    own = torch.from_numpy(_owned_rows(L)).to(DEV)
    Y = torch.empty_like(ref)
    bad = 0
    for _ in range(40):
        Y.fill_(0)
        B.moe_dispatch_grouped_gemm(h, xd, Wd, Y)
        bad += int((Y.view(torch.int16)[own] != ref.view(torch.int16)[own]).any(dim=1).sum().item())
    assert h.status() == 0
    assert bad == 0, f"{bad} rows differed over 40 calls"


def _random_gemm_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        e = int(rng.choice([1, 2, 3, 7, 16, 64, 256]))
        k = int(rng.integers(1, min(e, 8) + 1))
        s = int(rng.integers(1, 1000))
        K = 8 * int(rng.integers(8, 81))       # 64 .. 640, any multiple of 8
        N = 8 * int(rng.integers(1, 81))       # 8 .. 640
        c = dict(s=s, e=e, k=k, K=K, N=N)
        r = rng.random()
        if r < 0.35:
            c["capacity"] = int(rng.integers(1, max(2, 2 * s * k // e)))
            if rng.random() < 0.4:
                c["priority"] = "kmajor"
        elif r < 0.6:
            c["pad"] = int(rng.choice([8, 64, 128, 256]))
        out.append(c)
    return out


@pytest.mark.parametrize("case", _random_gemm_cases(20, seed=1202),
                         ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_random_shapes_match_float64_and_fused_is_identical(case):
    """Seeded random layouts and K, N (any multiples of 8): the plain GEMM
    against a float64 matmul per segment, the fused form bit for bit equal
    to it, rows no route owns untouched."""
    c = dict(case)
    s, e, k, K, N = (c.pop(n) for n in ("s", "e", "k", "K", "N"))
    h, x, X, OX, L = _setup(s, e, k, K, seed=s + K, **c)
    g = torch.Generator().manual_seed(N)
    Wt = (torch.randn(e, N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    Wd = Wt.to(DEV)
    Y = B.moe_grouped_gemm(h, X, Wd, _sentinel_out(h.rows, N))
    Yf = B.moe_dispatch_grouped_gemm(h, x.to(DEV), Wd, _sentinel_out(h.rows, N))
    torch.cuda.synchronize()
    assert h.status() == 0
    _check_float64(Y, OX, Wt, L)
    np.testing.assert_array_equal(bits(Yf), bits(Y))
    _check_unowned_untouched(Y, L)
