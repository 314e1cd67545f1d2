"""Seeded synthetic workloads for the MoE token path.

This module draws inputs only: it holds no step of the method (no gating,
no layout, no dispatch or combine arithmetic).  The tests feed what it draws
to both the CUDA library and the CPU oracle, and the benchmark times the
library on it.  It imports nothing else from the package.

Shapes follow the workloads the pages measure (no trained weights or
routing traces are available, so N(0, 1) router logits stand in for them):

* ``tiny-capacity``        s=256   m=128  e=8   k=2  fp32, capacity 80 (cf 1.25)
* ``mixtral-dropless``     s=8192  m=4096 e=8   k=2  bf16, dropless
* ``fine-grained-skewed``  s=16384 m=4096 e=128 k=8  bf16, dropless, Zipf-like
  expert bias b_j = 1.5*log(1/(j+1)), dedup counts over 8 virtual ranks
* ``diffusiongemma-replay`` s=2791 m=2816 e=128 k=8 bf16, dropless; 30 layers x
  3 passes, one seed per (pass, layer)
* ``gshard-capacity``      s=32768 m=2048 e=64  k=6  bf16, capacity 3072 (cf 1.0),
  expert bias b_j = -1.2*log(j+1) (the log of a Zipf(1.2) weight)

Draw order per seed: logits, x, y (expert output, dispatched shape), dout.
The logits always come from the CPU generator (the routing of a seed is the
same on every device); on a GPU the payloads come from that device's
generator.  bf16 tensors are fp32 N(0, 1) draws rounded to nearest-even.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    s: int            # tokens
    m: int            # hidden size
    e: int            # experts
    k: int            # routes per token
    dtype: str        # "f32" or "bf16" (activations; logits and gates are fp32)
    capacity: int     # slots per expert; 0 = dropless grouped layout
    R: int            # virtual ranks for the dedup counts; 0 = none
    seed: int
    zipf_alpha: float = 0.0   # expert bias b_j = -alpha * log(j + 1)
    renorm: int = 1
    layers: int = 1
    passes: int = 1

    @property
    def rows(self) -> int:
        """Rows of the dispatched buffer: e*capacity, or s*k when dropless."""
        return self.e * self.capacity if self.capacity > 0 else self.s * self.k

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny-capacity", s=256, m=128, e=8, k=2, dtype="f32", capacity=80, R=0, seed=0),
        Workload("mixtral-dropless", s=8192, m=4096, e=8, k=2, dtype="bf16", capacity=0, R=0, seed=2),
        Workload("fine-grained-skewed", s=16384, m=4096, e=128, k=8, dtype="bf16", capacity=0, R=8,
                 seed=3, zipf_alpha=1.5),
        Workload("diffusiongemma-replay", s=2791, m=2816, e=128, k=8, dtype="bf16", capacity=0, R=0,
                 seed=4000, layers=30, passes=3),
        Workload("gshard-capacity", s=32768, m=2048, e=64, k=6, dtype="bf16", capacity=3072, R=0,
                 seed=5, zipf_alpha=1.2),
    ]
}


def replay_seed(w: Workload, pass_id: int, layer: int) -> int:
    """Seed of one (pass, layer) call of the stacked-replay workload."""
    return w.seed + 100 * pass_id + layer


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_logits(w: Workload, device="cpu", seed: int | None = None) -> torch.Tensor:
    """Router logits [s,e] f32, drawn on the CPU whatever the device, so a seed
    gives the same routing everywhere (plus the workload's expert bias)."""
    g = _gen("cpu", w.seed if seed is None else seed)
    logits = torch.randn(w.s, w.e, generator=g, dtype=torch.float32)
    if w.zipf_alpha:
        bias = torch.tensor([-w.zipf_alpha * math.log(j + 1) for j in range(w.e)], dtype=torch.float32)
        logits += bias
    return logits.to(device)


def make_inputs(w: Workload, device="cpu", seed: int | None = None, with_grad: bool = True,
                rows: int | None = None) -> dict:
    """Draw logits [s,e] f32, x [s,m], y [rows,m] and dout [s,m] from one seed
    (rows defaults to the workload's; a padded layout needs more).  The
    logits come first from the seed's CPU generator, so the routing is the
    same on every device; the payloads continue on the device's generator
    (on the CPU that is the same generator, so a CPU draw is one stream)."""
    seed = w.seed if seed is None else seed
    g = _gen("cpu", seed)
    logits = torch.randn(w.s, w.e, generator=g, dtype=torch.float32)
    if w.zipf_alpha:
        bias = torch.tensor([-w.zipf_alpha * math.log(j + 1) for j in range(w.e)], dtype=torch.float32)
        logits += bias
    logits = logits.to(device)
    if torch.device(device).type != "cpu":
        g = _gen(device, seed)
    dt = w.torch_dtype
    x = torch.randn(w.s, w.m, generator=g, device=device, dtype=torch.float32).to(dt)
    out = dict(logits=logits, x=x)
    if with_grad:
        out["y"] = torch.randn(w.rows if rows is None else rows, w.m, generator=g, device=device,
                               dtype=torch.float32).to(dt)
        out["dout"] = torch.randn(w.s, w.m, generator=g, device=device, dtype=torch.float32).to(dt)
    return out


def random_gates(s: int, k: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Positive, non-uniform weights [s,k] f32 for op-level combine checks."""
    g = _gen(device, seed)
    return torch.rand(s, k, generator=g, device=device, dtype=torch.float32) + 0.05


def random_routes(s: int, e: int, k: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """k distinct experts per token, uniformly at random, as int32 [s,k]."""
    g = _gen("cpu", seed)
    idx = torch.argsort(torch.rand(s, e, generator=g), dim=1)[:, :k].to(torch.int32)
    return idx.to(device)
