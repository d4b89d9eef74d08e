"""Host logic of bench.py's multi-rank path (independent replicas), on CPU with gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, lr, w = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + r, w)        # the slowest rank's time decides
    tot = bench.sum_over_ranks(16384, w)          # tokens of all replicas
    q.put((r, lr, w, mx, tot))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[0] for r in res] == [0, 1]
    assert all(r[2] == 2 and r[3] == 11.0 and r[4] == 32768 for r in res)


def test_reference_arm_under_two_ranks_prints_once():
    """torchrun-style launch of the reference arm: rank 0 prints one JSON line, rank 1 exits 0 silently."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "mid"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("workload", ["linear", "linear_peaked"])
def test_reference_arm_linear_workloads(workload):
    """The reference arm on the linear workloads (a small vocabulary): one JSON line with the
    arm's metric, the oracle as the timed program and a stated sample."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
           "--vocab", "256", "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"].startswith("fused linear-CE") and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and "sampled rows" in d["config"]["workload"]
    assert ("gradient filtering" in d["metric"]) == (workload == "linear_peaked")
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_linear_cpu_baseline_host_logic():
    """The linear line's cpu_baseline: the oracle on a bounded row sample, rows / seconds."""
    sys.path.insert(0, ROOT)
    import bench
    import gen
    p = gen.linear_custom(64, 32, 300, seed=41, n_ignore=3)
    b = bench.cpu_oracle_baseline_linear(p, budget_s=2.0, max_rows=8)
    assert b["kind"] == "oracle" and b["value"] > 0 and b["cores"] >= 1
    assert b["sample"].startswith("8 random rows")
