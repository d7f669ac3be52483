"""The bench's N > 1 path on CPU: world size 2 over gloo (no GPU).

The path shards by sequence and exchanges nothing on the data path: ranks run
replicas and only the timing is combined (max of the times, sum of the tokens).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init("gloo")
    w, r, _ = bench.dist_env()
    mx = bench.reduce_max(float(r + 1) * 1.5, dist, "cpu")
    sm = bench.reduce_sum(float(r + 1), dist, "cpu")
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "max": mx, "sum": sm}, f)
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks(tmp_path):
    """Max over ranks of the timed region and sum of the tokens, as bench.py combines replicas."""
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        d = json.load(open(tmp_path / f"rank{r}.json"))
        assert d == {"world": 2, "rank": r, "max": 3.0, "sum": 3.0}


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched on two ranks: rank 0 alone times the oracle and prints
    one JSON line; the other rank exits 0 without work."""
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.2",
           "--oracle-step-seconds", "0.3"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
