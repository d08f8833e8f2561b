"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The operator shards with no exchange, so N GPUs run N independent replicas
(weak scaling); the only cross-rank steps are the barrier and the max over
ranks of the step time, and the job's throughput is N x one problem's work
over that time.  No GPU is touched.
"""

import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dist.barrier()
        # rank r's step takes 10 + 7 r ms: the job takes the slowest
        ms = bench.max_over_ranks(10.0 + 7.0 * rank, dist, "cpu")
        value = bench.job_tflops(2e12, world, ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms} {value}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        ms, value = (float(v) for v in open(tmp_path / f"rank{r}.txt").read().split())
        assert ms == 17.0
        assert value == pytest.approx(world * 2e12 / 17e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of `bench.py --impl reference` exits 0 without output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""
