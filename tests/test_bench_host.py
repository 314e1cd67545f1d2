"""Host-side pieces of bench.py that need no GPU: the byte model, the
max-over-ranks aggregation on a two-process gloo group, and the reference
arm's rank behaviour under a multi-process launch."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from combine_moe_topk_gb300 import workloads as W  # noqa: E402


def test_byte_model_of_the_mixtral_like_step():
    w = W.WORKLOADS["mixtral-dropless"]
    b = bench.step_bytes(w, kept=w.s * w.k, u=w.s)
    x = w.s * w.m * 2  # 67,108,864
    assert x == 67108864
    # dispatch: x once + 2x written (+ the row indices); combine: 2x read + x written (+ rows, gates)
    assert b["dispatch"] == 3 * x + w.s * w.k * 4
    assert b["combine"] == 3 * x + w.s * w.k * 8
    assert b["combine_bwd"] == 5 * x + w.s * w.k * 12
    assert b["dispatch_bwd"] == 3 * x + w.s * w.k * 4
    assert bench.payload_bytes(w, w.s * w.k, w.s) == {"dispatch": 3 * x, "combine": 3 * x}


def test_byte_model_of_the_fused_backward_and_the_step():
    """The fused combine + gate backward moves the combine backward's bytes
    plus the expert ids read and the router gradient written; the fused gate
    + layout the two ops' bytes less the ids read back; a step counts each
    op it runs once (not the separate ops as well)."""
    w = W.WORKLOADS["fine-grained-skewed"]
    b = bench.step_bytes(w, kept=w.s * w.k, u=w.s)
    assert b["combine_gate_bwd"] == b["combine_bwd"] + w.s * w.k * 4 + w.s * w.e * 4
    assert b["gate_layout"] == b["topk_gate"] + b["layout"] - w.s * w.k * 4  # the ids are not read back
    assert bench.step_sum(b) == sum(b[op] for op in
                                    ("gate_layout", "dispatch", "combine", "combine_gate_bwd", "dispatch_bwd"))
    wn = W.WORKLOADS["tiny-capacity"].replace(renorm=0)
    bn = bench.step_bytes(wn, kept=100, u=60)
    assert bn["combine_gate_bwd"] == bn["combine_bwd"] + wn.s * wn.k * 4 + 2 * wn.s * wn.e * 4


def test_byte_model_counts_the_capacity_zero_tail():
    w = W.WORKLOADS["gshard-capacity"]
    kept, u = 150000, 30000
    b = bench.step_bytes(w, kept, u)
    rows_bytes = w.e * w.capacity * w.m * 2
    assert b["dispatch"] == u * w.m * 2 + rows_bytes + w.s * w.k * 4


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 3.0 - rank]
    got = bench.max_over_ranks(local, dist)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 3.0]
    assert bench.job_gbs(2, 1_000_000_000, 1.0) == pytest.approx(2000.0)
    assert bench.max_over_ranks([1.5], None) == [1.5]


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1",
                        "--warmup", "1", "--workload", "tiny-capacity", "--ref-seconds", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--workload", "tiny-capacity", "--ref-seconds", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_is_per_workload_and_tied_to_the_source(tmp_path):
    sha = bench.source_sha("combine_bwd")
    rec = {"wl-a": {"combine_bwd": {"dram_bytes_per_launch": 100, "source_sha": sha}},
           "wl-b": {"combine_bwd": {"dram_bytes_per_launch": 200, "source_sha": sha},
                    "combine": {"dram_bytes_per_launch": 300, "source_sha": "0" * 16}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    assert bench.traffic_record("combine_bwd", "wl-a", str(path))["dram_bytes_per_launch"] == 100
    assert bench.traffic_record("combine_bwd", "wl-b", str(path))["dram_bytes_per_launch"] == 200
    assert bench.traffic_record("combine_bwd", "no-such-workload", str(path)) is None
    assert bench.traffic_record("combine", "wl-b", str(path)) is None  # taken on another source
    # the committed record file parses and keys by workload
    committed = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    assert "fine-grained-skewed" in committed and "combine_gate_bwd" in committed["fine-grained-skewed"]


def test_gpus_flag_must_match_the_process_count():
    """--gpus N under a launcher that started a different number of ranks is
    refused instead of silently reporting one replica."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1", "--workload", "tiny-capacity", "--ref-seconds", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def test_gpus_flag_starts_one_process_per_gpu():
    """Without a launcher, --gpus 2 starts two ranks itself (torch.distributed.run
    on 127.0.0.1); the reference arm then prints one line, from rank 0."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                           "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1", "--workload", "tiny-capacity", "--ref-seconds", "1"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
