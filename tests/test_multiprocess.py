"""The multi-process (N > 1) paths of bench.py on CPU: two gloo ranks agree on
the slowest rank's time and the whole-job throughput, and the reference arm
under torchrun runs on rank 0 alone (one JSON line, every rank exits 0). The
decode itself shards as independent replicas (no collective on the data path),
so these host-side pieces are what the N > 1 runs add."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.reduce_max(10.0 + 5.0 * rank, dist)  # rank 1 is the slower one
    val = bench.whole_job_tflops(1e12, 4, world, ms / 1e3)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, val))


def test_gloo_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    # 2 ranks x 4 units x 1 TFLOP in 15 ms
    assert all(abs(g[2] - 2 * 4 / 0.015) < 1e-9 for g in got)


def test_reduce_max_without_a_process_group():
    import bench
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_tflops(2e12, 3, 1, 1.5) == 4.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the line carries every key of the bench contract
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["steps"] == 1 and d["warmup"] == 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]
