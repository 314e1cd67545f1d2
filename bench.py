#!/usr/bin/env python
"""Benchmark of the MoE token path on GB300.

One step = one pass of the whole path over one batch of seeded synthetic
input: top-k gate + dispatch layout (one kernel) -> dispatch -> combine ->
combine backward (gate-scaled dispatch + gate gradient) with the gate
backward (router logits' gradient) in the same kernel -> dispatch backward,
all on the layout handle the step built.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, on a bounded sample

Prints ONE JSON line.  ``value`` = algorithmic HBM bytes of a step / device
time of a step (GB/s), inputs resident in HBM, the K steps timed back to
back with no events between kernels (as one CUDA graph of the step when it
can be captured, else eager calls; ``config.launch`` says which).  The
step's working set is several times the 129 MB L2, so no L2 flush is
inserted between steps.  Further keys:

- ``ops`` / ``roofline``: per-kernel durations from a separate loop with
  events around every call (each after a short GPU sleep, so the host's
  enqueue is not timed); the roofline is the dominant kernel's algorithmic
  bytes over its mean duration against the measured copy bandwidth, with
  its ncu DRAM traffic from ``profiles/ncu_traffic.json``;
- ``dispatch_combine``: the pair as a CUDA graph on one handle, replayed
  back to back (the cached-replay case);
- ``replay``: the step on a saved handle (gate recomputed, no layout), and
  the layout launches seen meanwhile (must be 0);
- the step's handle is created once and rebuilt in place by each step's
  fused gate + layout kernel (no allocation or memset per step);
- ``routing``: drop fraction, and the dedup ratio over virtual ranks;
- ``e2e``: the same metric with every step's inputs copied from pinned
  host memory and its results copied back inside the timed region;
- ``expert_gemm``: the grouped GEMM consuming the dispatched rows, plain
  and fused with the dispatch, in TFLOP/s against the longer of its FLOP and
  weight-streaming bounds (outside ``value``);
- ``expert_parallel`` (workloads with virtual ranks): the expert-parallel
  layer's per-rank kernels, R ranks emulated on this GPU, per phase
  (outside ``value``; the exchange between GPUs is not measured here);
- ``cpu_baseline``: the oracle on the host's cores (and on one core).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine HBM GB/s and routed tokens/s on 1 GB300 vs HBM peak"
DEFAULT_WORKLOAD = "fine-grained-skewed"  # the largest workload: s=16384, m=4096, e=128, k=8
OPS = ["gate_layout", "dispatch", "combine", "combine_gate_bwd", "dispatch_bwd"]
KERNEL_FILE = {"topk_gate": "gate.cu", "layout": "layout.cu", "gate_layout": ("layout.cu", "gate.cu", "gate_core.cuh"),
               "dispatch": "dispatch.cu", "combine": "combine.cu",
               "combine_bwd": "combine.cu", "topk_gate_bwd": ("gate.cu", "router_grad.cuh"),
               "combine_gate_bwd": ("combine.cu", "router_grad.cuh"), "dispatch_bwd": "combine.cu"}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024  # GB300 L2 (a flush writes twice this)
SLEEP_CYCLES = 100_000  # ~50 us at 2 GHz: longer than the host's enqueue of one call
EP_SLEEP_CYCLES = 1_000_000  # ~0.5 ms: an expert-parallel phase enqueues several calls and allocations


# ------------------------------------------------------------ byte model --

def step_bytes(w, kept: int, u: int) -> dict:
    """Algorithmic HBM bytes of each op.  kept = kept routes, u = tokens with
    at least one kept route (both equal s*k and s when nothing is dropped)."""
    b, s, m, e, k = w.elem_bytes, w.s, w.m, w.e, w.k
    R = w.rows * m * b          # whole dispatched buffer (capacity: incl. the zero tail)
    x = s * m * b
    routes = s * k
    meta_r = routes * 4         # reading row[] (or idx)
    out = {
        "topk_gate": s * e * 4 + routes * 8,
        "layout": routes * 4 + routes * 13 + e * 12 + (s * w.R + w.R * 4 if w.R else 0),
        "dispatch": u * m * b + R + meta_r,
        "combine": kept * m * b + x + meta_r + routes * 4,
        "combine_bwd": x + kept * m * b + R + meta_r + routes * 8,
        "topk_gate_bwd": routes * 12 + s * e * 4 + (0 if w.renorm else s * e * 4),
        "dispatch_bwd": kept * m * b + x + meta_r,
    }
    # fused: the combine backward's bytes, plus the expert ids and the router
    # gradient written (and the logits without renorm); dgate is not re-read
    out["combine_gate_bwd"] = out["combine_bwd"] + routes * 4 + s * e * 4 + (0 if w.renorm else s * e * 4)
    # fused gate + layout: the gate's logits in and ids + gates out, the
    # layout's outputs; the ids are not read back
    out["gate_layout"] = out["topk_gate"] + out["layout"] - routes * 4
    return out


def step_sum(nbytes: dict) -> int:
    """Algorithmic bytes of one step: the ops the step runs."""
    return sum(nbytes[op] for op in OPS)


def payload_bytes(w, kept: int, u: int) -> dict:
    b, m = w.elem_bytes, w.m
    x = w.s * m * b
    R = w.rows * m * b
    return {"dispatch": u * m * b + R, "combine": kept * m * b + x}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s) for a kernel timed on its own."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def source_sha(op: str) -> str:
    """Hash of the kernel source file(s) of an op (ties a traffic record to it)."""
    files = KERNEL_FILE[op] if isinstance(KERNEL_FILE[op], tuple) else (KERNEL_FILE[op],)
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "combine_moe_topk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(op: str, workload: str, path: str | None = None):
    """Per-launch DRAM bytes of this op on this workload from the committed
    ncu summary, if it was taken on the kernel source as it is now (else
    None)."""
    path = path or os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload, {})
    except Exception:
        return None
    r = rec.get(op)
    if not r or r.get("source_sha") != source_sha(op):
        return None
    return r


def max_over_ranks(values, dist, device=None):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    job's time); identity without a process group."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            p = [x.strip() for x in l.split(",")]
            try:
                rows.append((float(p[0]), float(p[1]), p[4:8], p[3]))
            except Exception:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------- our arm -----

def run_ours(args, rank: int, world: int, dist):
    import torch

    from combine_moe_topk_gb300 import binding as B
    from combine_moe_topk_gb300 import workloads as W

    w = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    B.lib()
    dt = w.torch_dtype

    def buffers(seed):
        inp = W.make_inputs(w, device=dev, seed=seed)
        return dict(
            logits=inp["logits"], x=inp["x"], y=inp["y"], dout=inp["dout"],
            X=torch.empty(w.rows, w.m, dtype=dt, device=dev), out=torch.empty(w.s, w.m, dtype=dt, device=dev),
            dY=torch.empty(w.rows, w.m, dtype=dt, device=dev), dx=torch.empty(w.s, w.m, dtype=dt, device=dev),
            idx=torch.empty(w.s, w.k, dtype=torch.int32, device=dev),
            gate=torch.empty(w.s, w.k, dtype=torch.float32, device=dev),
            dgate=torch.empty(w.s, w.k, dtype=torch.float32, device=dev),
            dlogits=torch.empty(w.s, w.e, dtype=torch.float32, device=dev))

    S = buffers(w.seed + 1000 * rank)
    # the layout handle: created once (its memory allocated and zeroed), then
    # rebuilt in place by every step's gate + layout, with no allocation
    H = {0: B.moe_layout_create(w.s, w.e, w.k, w.capacity, w.R, device=dev)}

    pad = getattr(torch.cuda, "_sleep", None)

    def step(b=S, ev=None, slot=0):
        """One pass of the path on a layout handle rebuilt from this step's
        logits: the top-k gate fused into the layout build, dispatch,
        combine, the combine backward with the gate backward fused in, and
        the dispatch backward.  With ev (pairs of events per op), each op is
        bracketed by its own events, preceded by a short GPU sleep so that
        the host has enqueued the op before the start event is reached: the
        pair then times the kernel, not the host's launch overhead."""
        def mark(i, j):
            if ev is not None:
                if j == 0 and pad is not None:
                    pad(SLEEP_CYCLES)
                ev[i][j].record()

        h = H[slot]
        mark(0, 0)
        B.moe_topk_gate_layout(h, b["logits"], w.renorm, b["idx"], b["gate"])
        mark(0, 1)
        mark(1, 0)
        B.moe_dispatch(h, b["x"], b["X"])
        mark(1, 1)
        mark(2, 0)
        B.moe_combine(h, b["y"], b["gate"], b["out"])
        mark(2, 1)
        mark(3, 0)
        B.moe_combine_gate_bwd(h, b["dout"], b["gate"], b["y"], b["logits"], w.renorm, b["dY"], b["dgate"],
                               b["dlogits"])
        mark(3, 1)
        mark(4, 0)
        B.moe_dispatch_bwd(h, b["dY"], b["dx"])
        mark(4, 1)
        return h

    # kept routes / sending tokens for the byte model (outside any timing)
    h = step()
    drop = h.drop()
    kept = int((drop == 0).sum().item())
    u = int((drop == 0).any(dim=1).sum().item())
    rank_sum = int(h.rank_counts().sum().item()) if w.R else 0
    assert h.status() == 0, "device status after the first step"
    nbytes = step_bytes(w, kept, u)
    step_total = step_sum(nbytes)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # the step as one CUDA graph (replays skip the per-call host work); eager if capture fails
    graph, launch_mode, graph_launches = None, "eager", 0
    if not args.eager:
        try:
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for _ in range(2):
                    step()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            c0 = sum(B.moe_launch_count(i) for i in range(len(B.KERNELS)))
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            graph_launches = sum(B.moe_launch_count(i) for i in range(len(B.KERNELS))) - c0
            graph.replay()
            torch.cuda.synchronize()
            launch_mode = "cuda graph of the step (replayed)"
        except Exception as exc:  # capture unsupported here: time the eager path
            graph = None
            launch_mode = f"eager (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    for _ in range(args.warmup):
        run_step()
    barrier()

    # ---- the timed region: exactly K steps ---------------------------------
    # A step whose working set exceeds twice the L2 leaves nothing useful in
    # it for the next step: the K steps run back to back with no events
    # between them.  A smaller one would run from L2, so each step is timed
    # on its own after a write of more than the L2 (outside its events).
    K = args.steps
    flush = None if step_total >= 2 * L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    launches0 = [B.moe_launch_count(i) for i in range(len(B.KERNELS))]
    with ClockSampler(dev.index) as clk:
        barrier()
        elapsed_ms = time_loop(run_step, K, flush) * K
        barrier()
    launches = sum(B.moe_launch_count(i) - launches0[i] for i in range(len(B.KERNELS)))
    if graph is not None:
        launches = graph_launches * K

    if args.only_step:
        elapsed_ms = max_over_ranks([elapsed_ms], dist, dev)[0]
        if rank != 0:
            return None
        ms = elapsed_ms / K
        return {"metric": METRIC, "value": round(job_gbs(world, step_total, ms), 1), "unit": "GB/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": {"workload": w.name, "launch": launch_mode, "legs": "step only (profiling run)"},
                "gpu_launches": launches, "clocks": clk.summary()}

    # ---- per-kernel durations: events around each call, eager, own loop -----
    Kr = max(3, min(K, 200))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in OPS] for _ in range(Kr)]
    for i in range(Kr):
        step(ev=evs[i])
    torch.cuda.synchronize()
    samples = {op: sorted(evs[i][j][0].elapsed_time(evs[i][j][1]) for i in range(Kr)) for j, op in enumerate(OPS)}
    per_op = {op: statistics.mean(v) for op, v in samples.items()}
    spread = {op: (v[len(v) // 10], v[len(v) // 2], v[(9 * len(v)) // 10]) for op, v in samples.items()}

    # ---- dispatch + combine in steady state: a graph of the pair on one
    # handle (the cached-replay case), replayed back to back -----------------
    dc = run_dispatch_combine(w, S, dev, K)

    # ---- the recompute: the whole step on a saved handle, no layout --------
    rp = run_replay_step(w, S, dev, K)

    # ---- end to end: pinned host inputs in, results out, every step ----------
    e2e = run_e2e(w, S, step, buffers, dev, max(3, min(K, 50)), args.warmup)

    # ---- the tensor-core consumer of the dispatched rows (outside value) ------
    gemm = None if args.no_gemm else run_expert_gemm(w, S, dev)

    # ---- the expert-parallel layer's per-rank kernels (outside value) --------
    epl = run_expert_parallel(w, dev) if (w.R and not args.no_ep) else None

    elapsed_ms, e2e["ms"], dc["ms"], rp["ms"] = max_over_ranks([elapsed_ms, e2e["ms"], dc["ms"], rp["ms"]], dist,
                                                               dev)
    if rank != 0:
        return None

    ms_per_step = elapsed_ms / K
    value = job_gbs(world, step_total, ms_per_step)
    peak, peak_src = peaks()
    dom = max(per_op, key=per_op.get)
    achieved = nbytes[dom] / (per_op[dom] * 1e-3) / 1e9
    tr = traffic_record(dom, w.name)
    pay = payload_bytes(w, kept, u)
    dc_ms = dc["ms"]
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) router logits and activations (no trained weights or routing traces)",
        "config": {
            "workload": w.name, "s": w.s, "m": w.m, "e": w.e, "k": w.k,
            "mode": f"capacity {w.capacity}" if w.capacity else "dropless", "virtual_ranks": w.R,
            "step": "topk_gate+layout+dispatch+combine+combine_gate_bwd (combine backward with the gate backward "
                    "fused in)+dispatch_bwd on the step's handle",
            "launch": launch_mode,
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": (f"no flush: step working set {round(step_total / 1e6)} MB algorithmic, over twice the 129 MB L2"
                   if flush is None else
                   f"L2 flushed before every step (a {2 * L2_BYTES >> 20} MiB write, outside the timing): step "
                   f"working set {round(step_total / 1e6, 2)} MB; steps timed one by one"),
        },
        "routed_tokens_per_s": round(world * w.s * w.k / (ms_per_step * 1e-3), 1),
        "dispatch_combine": {
            "us": round(dc_ms * 1e3, 2), "how": dc["how"],
            "sum_of_op_events_us": round((per_op["dispatch"] + per_op["combine"]) * 1e3, 2),
            "gbs": round((nbytes["dispatch"] + nbytes["combine"]) / (dc_ms * 1e-3) / 1e9, 1),
            "payload_gbs": round((pay["dispatch"] + pay["combine"]) / (dc_ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round((nbytes["dispatch"] + nbytes["combine"]) / (dc_ms * 1e-3) / 1e9 / peak, 4),
            "routed_tokens_per_s": round(w.s * w.k / (dc_ms * 1e-3), 1),
        },
        "ops": {op: {"us": round(per_op[op] * 1e3, 2), "bytes": nbytes[op],
                     "gbs": round(nbytes[op] / (per_op[op] * 1e-3) / 1e9, 1),
                     "us_p10_p50_p90": [round(x * 1e3, 2) for x in spread[op]]} for op in OPS},
        "ops_note": f"per-kernel times from events around each call, eager, {Kr} separate steps, each call "
                    f"after a {SLEEP_CYCLES}-cycle GPU sleep so the events bracket the kernel"
                    + ("" if pad is not None else " (sleep unavailable: host gaps included)"),
        "roofline": {
            "kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (copy bandwidth)",
            "traffic": (tr["dram_bytes_per_launch"] if tr else None),
            "traffic_note": (tr.get("note") if tr else "no ncu capture of this kernel source on this workload"),
            "algorithmic_bytes": nbytes[dom],
        },
        "e2e": {"value": round(job_gbs(world, step_total, e2e["ms"]), 1), "unit": "GB/s",
                "ms_per_step": round(e2e["ms"], 4), "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "steps": e2e["steps"], "how": e2e["how"]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "kept_routes": kept,
        "sending_tokens": u,
        "routing": {
            "drop_fraction": round(1.0 - kept / (w.s * w.k), 6),
            **({"dedup": {"rank_counts_sum": rank_sum, "routes_per_sent_token": round(kept / rank_sum, 4),
                          "virtual_ranks": w.R}} if w.R and rank_sum else {}),
        },
        "replay": {
            "ms_per_step": round(rp["ms"], 5), "full_step_ms": round(ms_per_step, 5),
            "saved_fraction": round(1.0 - rp["ms"] / ms_per_step, 4),
            "layout_launches_during": rp["layout_launches"], "how": rp["how"],
        },
    }
    if gemm is not None:
        line["expert_gemm"] = gemm
    if epl is not None:
        line["expert_parallel"] = epl
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args)
    return line


def time_loop(run, n: int, flush=None) -> float:
    """Mean device time (ms) of n calls of run(): back to back between two
    events, or, with a flush buffer (a working set that L2 would hold), each
    call timed on its own after a write of that buffer."""
    import torch

    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            run()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush.fill_(1)
        a.record()
        run()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n


def small_working_set(w) -> bool:
    """Whether a step's inputs and outputs would stay in L2 between steps."""
    return step_sum(step_bytes(w, w.s * w.k, w.s)) < 2 * L2_BYTES


def run_dispatch_combine(w, S, dev, K: int):
    """Dispatch + combine on one handle, as a CUDA graph of the pair replayed
    K times back to back (events around the whole loop): the steady-state
    time of the pair with no host work between kernels.  Inputs and outputs
    of one pair (x, X, y, out) exceed the 129 MB L2 for every workload but
    the smallest, so no flush is inserted."""
    import torch

    from combine_moe_topk_gb300 import binding as B

    h = B.moe_dispatch_layout(S["idx"], w.e, w.capacity, w.R)
    torch.cuda.synchronize()

    def pair():
        B.moe_dispatch(h, S["x"], S["X"])
        B.moe_combine(h, S["y"], S["gate"], S["out"])

    how = "graph of dispatch + combine on one handle"
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            pair()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pair()
        run = g.replay
    except Exception as exc:
        run, how = pair, f"eager calls (graph capture failed: {type(exc).__name__})"
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    n = max(5, min(K, 500))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if small_working_set(w) else None
    ms = time_loop(run, n, flush)
    assert h.status() == 0
    h.destroy()
    how += ", each replay timed alone after an L2 flush" if flush is not None else ", replayed back to back"
    return {"ms": ms, "how": f"{how}, {n} pairs"}


def run_replay_step(w, S, dev, K: int):
    """The activation-checkpoint recompute of one step: the same kernels as
    the step (the gate is recomputed, routing pinned) on a handle built
    before the timed region, so no layout kernel runs.  A CUDA graph of it,
    replayed back to back; the layout launch counter must not move."""
    import torch

    from combine_moe_topk_gb300 import binding as B

    h = B.moe_dispatch_layout(S["idx"], w.e, w.capacity, w.R)
    torch.cuda.synchronize()

    def again():
        B.moe_topk_gate(S["logits"], w.k, w.renorm, S["idx"], S["gate"])
        B.moe_dispatch(h, S["x"], S["X"])
        B.moe_combine(h, S["y"], S["gate"], S["out"])
        B.moe_combine_gate_bwd(h, S["dout"], S["gate"], S["y"], S["logits"], w.renorm, S["dY"], S["dgate"],
                               S["dlogits"])
        B.moe_dispatch_bwd(h, S["dY"], S["dx"])

    how = "graph of the step on a saved handle (gate recomputed, no layout)"
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            again()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            again()
        run = g.replay
    except Exception as exc:
        run, how = again, f"eager calls (graph capture failed: {type(exc).__name__})"
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    layouts = B.moe_launch_count("layout") + B.moe_launch_count("gate_layout")
    n = max(5, min(K, 500))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if small_working_set(w) else None
    ms = time_loop(run, n, flush)
    moved = B.moe_launch_count("layout") + B.moe_launch_count("gate_layout") - layouts
    assert h.status() == 0
    h.destroy()
    how += ", each replay timed alone after an L2 flush" if flush is not None else ", replayed back to back"
    return {"ms": ms, "layout_launches": moved, "how": f"{how}, {n} steps"}


def run_expert_gemm(w, S, dev, reps: int = 10):
    """The grouped-GEMM consumer of the dispatched rows (not part of the step
    or of ``value``): synthetic expert weights W [e, N, m], N = m, bf16.
    Times dispatch, the grouped GEMM on the dispatched rows, and the fused
    dispatch + GEMM that gathers the token rows itself (CUDA events, one
    call each, the three in turn, median of ``reps``; the SM clocks seen)."""
    import torch

    from combine_moe_topk_gb300 import binding as B

    if w.dtype != "bf16" or w.m % 256:
        return {"skipped": "the tensor-core GEMM takes bf16 rows with m a multiple of 256"}
    N = w.m
    g = torch.Generator(device=dev).manual_seed(w.seed + 77)
    Wt = (torch.randn(w.e, N, w.m, device=dev, generator=g) * w.m ** -0.5).to(torch.bfloat16)
    h = B.moe_dispatch_layout(S["idx"], w.e, w.capacity, w.R)
    X = torch.empty(h.rows, w.m, dtype=torch.bfloat16, device=dev)
    Y = torch.empty(h.rows, N, dtype=torch.bfloat16, device=dev)
    kept = int(h.counts().sum().item())

    # the three calls take turns within each repetition, so that the GPU's
    # warming (and its power cap) over the block weighs on each alike
    calls = [lambda: B.moe_dispatch(h, S["x"], X), lambda: B.moe_grouped_gemm(h, X, Wt, Y),
             lambda: B.moe_dispatch_grouped_gemm(h, S["x"], Wt, Y)]
    for fn in calls:
        for _ in range(2):
            fn()
    ts = [[], [], []]
    with ClockSampler(dev.index) as clk:
        for _ in range(reps):
            for i, fn in enumerate(calls):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                ts[i].append(a.elapsed_time(b))
    t_d, t_g, t_f = (statistics.median(t) for t in ts)
    assert h.status() == 0
    h.destroy()
    flops = 2.0 * kept * w.m * N
    peak, src = bf16_peak()
    hbm, hsrc = peaks()
    tf = lambda ms: flops / (ms * 1e-3) / 1e12
    # the bytes a GEMM must move at least: its rows in, every expert's weights
    # once, its outputs; with many experts and few rows each, streaming the
    # weights takes longer than the MMAs
    gemm_bytes = kept * w.m * 2 + w.e * N * w.m * 2 + kept * N * 2
    t_tensor = flops / (peak * 1e12)
    t_hbm = gemm_bytes / (hbm * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    t_bound_ms = max(t_tensor, t_hbm) * 1e3
    return {
        "N": N, "K": w.m, "rows": int(Y.shape[0]), "kept_rows": kept, "flops": flops, "min_bytes": gemm_bytes,
        "us_dispatch": round(t_d * 1e3, 1), "us_gemm": round(t_g * 1e3, 1),
        "us_fused_dispatch_gemm": round(t_f * 1e3, 1),
        "tflops_gemm": round(tf(t_g), 1), "tflops_fused": round(tf(t_f), 1),
        "tflops_dispatch_then_gemm": round(tf(t_d + t_g), 1),
        "roofline": {"bound": bound, "peak": peak, "unit": "TFLOP/s",
                     "peak_source": f"{src} bf16 dense (burst, kernel timed alone)",
                     "hbm_peak_gbs": hbm, "hbm_peak_source": hsrc,
                     "us_at_bound": round(t_bound_ms * 1e3, 1),
                     "frac_gemm": round(tf(t_g) / peak, 4), "frac_fused": round(tf(t_f) / peak, 4),
                     "frac_of_bound_gemm": round(t_bound_ms / t_g, 4),
                     "frac_of_bound_fused": round(t_bound_ms / t_f, 4)},
        "clocks": clk.summary(),
        "note": "synthetic N(0,1)/sqrt(m) expert weights; events around single calls, the three calls "
                f"in turn, median of {reps}; not included in value; the bound is the longer of the FLOPs at "
                "the bf16 peak and min_bytes (rows in, each expert's weights once, outputs) at the copy "
                "bandwidth",
    }


def run_expert_parallel(w, dev, reps: int = 3):
    """The expert-parallel layer's per-rank kernels (outside value): R ranks
    of this workload (rank r's tokens from seed + r, experts [r*E, (r+1)*E)),
    all emulated on this GPU, forward and backward with an identity expert.
    Each phase of each rank is timed with events (median of reps); the
    all-to-alls between the ranks are device copies here, timed apart --
    the exchange between GPUs is not measured on one GPU."""
    import torch

    from combine_moe_topk_gb300 import binding as B
    from combine_moe_topk_gb300 import ep as EP
    from combine_moe_topk_gb300 import workloads as W

    R, E, b = w.R, w.e // w.R, w.elem_bytes
    srcs = []
    for r in range(R):
        inp = W.make_inputs(w, device=dev, seed=w.seed + r, with_grad=False)
        idx, gate = B.moe_topk_gate(inp["logits"], w.k, w.renorm)
        srcs.append(dict(x=inp["x"], idx=idx, gate=gate, dout=inp["x"]))  # the upstream gradient: any rows

    def a2a(bufs, plans, back=False):
        if not back:
            pieces = [torch.split(bufs[i], plans[i].send_counts) for i in range(R)]
            return [torch.cat([pieces[i][j] for i in range(R)]) for j in range(R)]
        pieces = [torch.split(bufs[j], plans[j].recv_counts) for j in range(R)]
        return [torch.cat([pieces[j][i] for j in range(R)]) for i in range(R)]

    times = {}
    pad = getattr(torch.cuda, "_sleep", None)

    def timed(name, fn):
        out = None
        ts = []
        for _ in range(reps):
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if pad is not None:
                pad(EP_SLEEP_CYCLES)  # the host enqueues the phase while the GPU sleeps
            a.record()
            out = fn()
            c.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(c))
        times.setdefault(name, []).append(statistics.median(ts))
        return out

    hs = [timed("layout", lambda r=r: B.moe_dispatch_layout_ex(srcs[r]["idx"], w.e, w.capacity, R, send_slots=True))
          for r in range(R)]
    counts = torch.stack([h.rank_counts() for h in hs]).cpu().tolist()
    routes = torch.stack([EP.route_counts(h) for h in hs]).cpu().tolist()
    plans = [EP.Plan([int(v) for v in counts[r]], [int(counts[i][r]) for i in range(R)],
                     [int(routes[i][r]) for i in range(R)]) for r in range(R)]
    sends = [timed("pack+send", lambda r=r: EP.source_send(hs[r], srcs[r]["x"], srcs[r]["gate"], plans[r]))
             for r in range(R)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rows = a2a([sd.X_send for sd in sends], plans)
    ids = a2a([sd.meta_idx for sd in sends], plans)
    gts = a2a([sd.meta_gate for sd in sends], plans)
    torch.cuda.synchronize()
    ex_fwd = time.perf_counter() - t0
    recvs = [timed("receive", lambda d=d: EP.dest_receive(rows[d], ids[d], gts[d], E, plans[d].routes_recv))
             for d in range(R)]
    P = [timed("partial", lambda d=d: EP.dest_partial(recvs[d], recvs[d].X)) for d in range(R)]
    Pb = a2a(P, plans, back=True)
    outs = [timed("reduce", lambda r=r: EP.source_reduce(hs[r], sends[r], Pb[r])) for r in range(R)]
    dPs = [timed("send_grad", lambda r=r: EP.source_send_grad(hs[r], sends[r], srcs[r]["dout"])) for r in range(R)]
    dP = a2a(dPs, plans)
    cb = [timed("combine_bwd", lambda d=d: EP.dest_combine_bwd(recvs[d], dP[d], recvs[d].X)) for d in range(R)]
    dgb = a2a([c[1] for c in cb], plans, back=True)
    timed_dg = [timed("dgate", lambda r=r: EP.source_dgate(hs[r], sends[r], dgb[r])) for r in range(R)]
    dxp = [timed("dispatch_bwd", lambda d=d: EP.dest_dispatch_bwd(recvs[d], cb[d][0])) for d in range(R)]
    dxb = a2a(dxp, plans, back=True)
    [timed("reduce_grad", lambda r=r: EP.source_reduce(hs[r], sends[r], dxb[r])) for r in range(R)]
    torch.cuda.synchronize()
    for h in hs + [rc.h for rc in recvs]:
        assert h.status() == 0
    sent = sum(sum(p.send_counts) for p in plans)
    nroutes = sum(p.routes_recv for p in plans)
    row = w.m * b
    # bytes per phase over all ranks: payload rows only (metadata is < 1 %)
    pb = {"pack+send": sum(w.s for _ in range(R)) * row + sent * row,
          "receive": sent * row + nroutes * row, "partial": nroutes * row + sent * row,
          "reduce": sent * row + R * w.s * row, "send_grad": R * w.s * row + sent * row,
          "combine_bwd": sent * row + 2 * nroutes * row, "dispatch_bwd": nroutes * row + sent * row,
          "reduce_grad": sent * row + R * w.s * row}
    per = {k: round(sum(v) * 1e3, 1) for k, v in times.items()}
    hbm, _ = peaks()
    return {
        "ranks": R, "experts_per_rank": E, "tokens_per_rank": w.s,
        "rows_sent": sent, "routes": nroutes, "routes_per_sent_row": round(nroutes / max(1, sent), 3),
        "us_per_phase_all_ranks": per,
        "gbs_per_phase": {k: round(pb[k] / (per[k] * 1e-6) / 1e9, 1) for k in pb if per.get(k)},
        "busiest_rank_routes": max(p.routes_recv for p in plans),
        "emulated_exchange_ms": round(ex_fwd * 1e3, 2),
        "how": f"{R} ranks emulated on one GPU, each phase of each rank timed alone after a GPU sleep (median of "
               f"{reps}), summed over "
               "ranks; identity expert; the all-to-all is a device copy here and the exchange between GPUs is "
               f"unmeasured; copy peak {hbm} GB/s",
    }


def run_e2e(w, S, step, buffers, dev, K, warmup):
    """Every step copies its inputs from pinned host memory to the device,
    runs the path and copies its results (out, dx, dgate) back.  Steps are
    pipelined over three streams (copy in, compute, copy out) with two
    device buffer sets, so step i+1's inputs travel while step i computes."""
    import torch

    sets = [S, buffers(w.seed + 7)]
    in_names = ("logits", "x", "y", "dout")
    out_names = ("out", "dx", "dlogits")
    h_in = [{n: sets[j][n].cpu().pin_memory() for n in in_names} for j in range(2)]
    h_out = [{n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype).pin_memory() for n in out_names}
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            j = i % 2
            b = sets[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[j])  # the set's previous step has read its inputs
                for name in in_names:
                    b[name].copy_(h_in[j][name], non_blocking=True)
                ev_in[j].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[j])
                if i >= 2:
                    s_cmp.wait_event(ev_out[j])  # its previous results have left
                step(b)
                ev_cmp[j].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[j])
                for name in out_names:
                    h_out[j][name].copy_(b[name], non_blocking=True)
                ev_out[j].record(s_out)

    run(max(2, warmup))
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_cmp.wait_event(t0)
    s_out.wait_event(t0)
    run(K)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_cmp)
    t1.record(s_in)
    torch.cuda.synchronize()
    return {"ms": t0.elapsed_time(t1) / K, "h2d": h2d, "d2h": d2h, "steps": K,
            "how": "pinned host -> device copies, the path, device -> host copies of out, dx, dlogits; "
                   "pipelined over copy-in / compute / copy-out streams, two buffer sets"}


# --------------------------------------------------------- oracle (CPU) --

def oracle_sample(w, s_sample: int):
    """Inputs of the first s_sample tokens of the workload, drawn on the CPU."""
    from combine_moe_topk_gb300 import workloads as W

    cap = 0
    if w.capacity:
        cap = max(1, -(-w.capacity * s_sample // w.s))  # same capacity factor on the sample
    ws = w.replace(s=s_sample, capacity=cap)
    return ws, W.make_inputs(ws)


def oracle_step(ws, inp):
    import numpy as np

    import oracle

    def nb(t):
        import torch

        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    arrs = {k: nb(v) for k, v in inp.items()}
    t0 = time.perf_counter()
    idx, gate = oracle.topk_gate(arrs["logits"], ws.k, ws.renorm)
    L = oracle.layout(idx, ws.e, ws.capacity, ws.R)
    oracle.dispatch(L["row"], arrs["x"], L["rows"])
    oracle.combine(L["row"], gate, arrs["y"])
    dY, dgate = oracle.combine_bwd(L["row"], gate, arrs["dout"], arrs["y"])
    oracle.topk_gate_bwd(arrs["logits"], idx, gate, dgate, ws.e, ws.renorm)
    oracle.dispatch_bwd(L["row"], dY)
    dt = time.perf_counter() - t0
    kept = int((L["drop"] == 0).sum())
    u = int((L["drop"] == 0).any(axis=1).sum())
    return dt, step_bytes(ws, kept, u)


def oracle_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, args):
    """The oracle, as it stands, on the host cores: whole steps of the full
    workload, repeated for about args.cpu_seconds of CPU work."""
    import oracle

    cores = oracle.set_threads(oracle_cores())
    ws, inp = oracle_sample(w, w.s)
    times, nbytes = [], None
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < args.cpu_seconds and len(times) < 100):
        dt, nbytes = oracle_step(ws, inp)
        times.append(dt)
    oracle.set_threads(1)
    per = statistics.median(times)
    # the same oracle on one core, a few steps (the parity authority's own speed)
    one, t_start = [], time.perf_counter()
    while not one or (time.perf_counter() - t_start < args.cpu_seconds / 2 and len(one) < 20):
        one.append(oracle_step(ws, inp)[0])
    per1 = statistics.median(one)
    return {"value": round(step_sum(nbytes) / per / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} full steps of {w.name} (s={w.s}, m={w.m}), median {per:.3f} s each",
            "single_core": {"value": round(step_sum(nbytes) / per1 / 1e9, 3), "unit": "GB/s", "cores": 1,
                            "sample": f"{len(one)} full steps, median {per1:.3f} s each"}}


def run_reference(args, rank: int, world: int):
    """The CPU oracle as the reference arm: each step is the whole path on the
    first s' tokens of the workload, s' sized so that warmup + steps take
    about args.ref_seconds in total."""
    if rank != 0:
        return None
    from combine_moe_topk_gb300 import workloads as W

    import oracle

    w = W.WORKLOADS[args.workload]
    cores = oracle.set_threads(oracle_cores())
    probe = min(w.s, 256)
    ws, inp = oracle_sample(w, probe)
    oracle_step(ws, inp)
    dt, _ = oracle_step(ws, inp)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    s_sample = int(max(32, min(w.s, probe * budget / max(dt, 1e-6))))
    ws, inp = oracle_sample(w, s_sample)
    for _ in range(args.warmup):
        oracle_step(ws, inp)
    times = []
    nbytes = None
    for _ in range(args.steps):
        dt, nbytes = oracle_step(ws, inp)
        times.append(dt)
    per = sum(times) / len(times)
    value = step_sum(nbytes) / per / 1e9
    sample = f"{ws.s} of {w.s} tokens of {w.name} (m={w.m}) per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) router logits and activations",
        "config": {"workload": w.name, "s": w.s, "m": w.m, "e": w.e, "k": w.k,
                   "mode": f"capacity {w.capacity}" if w.capacity else "dropless", "virtual_ranks": w.R,
                   "step": "topk_gate+layout+dispatch+combine+combine_bwd+topk_gate_bwd+dispatch_bwd (CPU oracle)"},
        "routed_tokens_per_s": round(ws.s * ws.k / per, 1),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def relaunch(n: int) -> int:
    """Run this command as n processes on one node (one per GPU) under
    torch.distributed.run; returns their exit status."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle work for cpu_baseline")
    ap.add_argument("--ref-seconds", type=float, default=120.0, help="total oracle work of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gemm", action="store_true", help="skip the expert_gemm figures")
    ap.add_argument("--no-ep", action="store_true", help="skip the expert_parallel figures")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of a CUDA graph of the step")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step alone: no per-op, pair, replay, end-to-end, GEMM or CPU legs (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start them (torchrun), each runs this file again
        sys.exit(relaunch(args.gpus))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one process per GPU")
    dist = None
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as td

            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            td.init_process_group("nccl")
            dist = td
        line = run_ours(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
