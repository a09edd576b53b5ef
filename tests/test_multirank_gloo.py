"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

Each rank runs an independent sequence; the only cross-rank steps are the
barrier and the max-over-ranks timing used for the whole-job throughput, and
the reference arm prints from rank 0 only.  No GPU needed."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank                      # rank 1 is the slower one
        mx = bench.max_over_ranks(ms, world, "cpu")
        out[rank] = (mx, bench.job_tflops(1e12, 4, world, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        mx, tf = res[r]
        assert mx == 150.0
        # 2 ranks x 4 steps x 1 TFLOP over the slowest rank's 150 ms
        assert tf == pytest.approx(2 * 4 * 1.0 / 0.150)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "c2", "--steps", "1", "--warmup", "1",
           "--cpu-seconds", "0.1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
