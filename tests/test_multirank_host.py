"""Host logic of the multi-GPU path, run as two gloo ranks on the CPU.

Under torchrun every rank of bench.py denoises its own canvas (independent
problems, no collective on the data path); the only cross-rank steps are the
barriers around the timed region and the max over ranks of the elapsed time,
from which rank 0 reports whole-job throughput.  These tests run those steps
with world size 2 over gloo (127.0.0.1) and check the reference arm's rank
gating.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # every rank times its own canvas; the job's time is the slowest rank's
        elapsed_ms = [12.5, 20.0][rank]
        results[rank] = bench.max_over_ranks(elapsed_ms, world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        assert dict(results) == {0: 20.0, 1: 20.0}


def test_whole_job_throughput_counts_all_ranks():
    # value = tokens of all ranks / max-over-ranks time (weak scaling: each rank its own canvas)
    tokens, steps, world, max_ms = 256, 100, 2, 20.0
    value = tokens * steps * world / (max_ms / 1e3)
    assert value == pytest.approx(2 * 256 * 100 / 0.02)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args, rank=1, world=2) is None


def test_single_rank_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
