"""The N > 1 path of bench.py on the CPU: two gloo ranks exercise the max-over-ranks
timing and the whole-job aggregation bench.py uses under torchrun, and a real
two-rank torchrun launch of the reference arm prints exactly one JSON line (rank 0)
while rank 1 exits cleanly without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.rank_max(local_ms[rank], world, "cpu")
        dist.barrier()
        out[rank] = (ms, bench.job_value(1000.0, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    local_ms = [3.0, 5.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), local_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 5.5  # both ranks see the slowest rank's time
        assert value == pytest.approx(1000.0 * world / 5.5e-3)  # whole job: both replicas' units


def test_single_rank_needs_no_process_group():
    import bench
    assert not dist.is_initialized()
    assert bench.rank_max(4.25, 1) == 4.25
    assert bench.job_value(845680, 1, 4.25) == pytest.approx(845680 / 4.25e-3)


def test_torchrun_two_ranks_reference_arm_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    for key in ("metric", "unit", "ms_per_step", "higher_is_better", "scaling", "config", "cpu_baseline", "e2e"):
        assert key in d
