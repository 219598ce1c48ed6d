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
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=120, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""
