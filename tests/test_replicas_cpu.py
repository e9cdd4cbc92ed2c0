"""The multi-GPU path is replicas only: each rank decodes its own batch and
bench.py reports the whole job's bytes over the slowest rank's time.  These
tests run that host logic as two gloo ranks on the CPU."""
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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [2.0, 5.0][rank]
    ms_max = bench.max_over_ranks(local_ms, world)
    gbs = bench.aggregate_gbs(1e9, world, ms_max)
    out[rank] = (ms_max, gbs)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms_max, gbs = out[rank]
        assert ms_max == 5.0                      # the slowest rank's time
        assert gbs == pytest.approx(2e9 / 5e-3 / 1e9)   # both ranks' bytes


def test_single_rank_helpers_need_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_gbs(553906176, 1, 0.1) == pytest.approx(5539.06176)


def test_reference_arm_prints_on_rank_zero_only():
    # under torchrun only rank 0 runs the (CPU) reference arm; other ranks exit 0
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
