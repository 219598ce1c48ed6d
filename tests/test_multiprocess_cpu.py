"""The N-replica path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py --gpus N runs N independent replicas (the path has no exchange step):
the whole-job value is the tokens all ranks processed over the slowest rank's
timed seconds, and only rank 0 prints.  These tests exercise that host logic
with world size 2 and no GPU."""
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


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r timed 1.5 + r seconds over 1000 * (r + 1) tokens
        t, n = bench.aggregate_over_ranks(1.5 + rank, 1000 * (rank + 1), "cpu", dist)
        out[rank] = (t, n)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_tokens():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time and the tokens of both
    assert res[0] == (2.5, 3000.0) and res[1] == (2.5, 3000.0)


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate_over_ranks(1.25, 4096, "cpu", None) == (1.25, 4096.0)


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the oracle arm; rank 1 prints nothing
    and exits 0 (no process group, no oracle work)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "0"], env=env,
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""


def test_gpus_must_match_the_launched_replicas():
    """--gpus N without N launched processes is refused before any work, so a
    line can never report a GPU count it did not time."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=120, cwd=ROOT)
    assert res.returncode != 0
    assert "WORLD_SIZE=1" in res.stderr


def test_torchrun_launch_of_two_reference_replicas():
    """The launch the driver uses for N > 1 (torch.distributed.run, one process
    per rank, 127.0.0.1): rank 0 alone prints one JSON line of the oracle arm,
    rank 1 exits 0.  On the small workload so that it takes seconds."""
    import json
    res = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--gpus", "2", "--workload", "tiny",
                          "--steps", "2", "--warmup", "0"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [x for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    # the measured seconds of the steps are what ms_per_step reports
    assert rec["ms_per_step"] * rec["steps"] <= rec["cpu_baseline"]["measured_s"] * 1e3 + 1e-6
