"""The N > 1 path of bench.py on CPU: world-size-2 gloo process groups.

Decode is sharded as independent replicas (sequences share nothing), so the
only cross-rank step is the timing: rank 0 reports the whole job's bytes over
the slowest rank's step time."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = [0.10, 0.25][rank]  # rank 1 is the slow one
        m = bench.max_over_ranks(step_ms, dist)
        dist.barrier()
        results[rank] = (m, bench.whole_job_gbs(545_891_164, world, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert got[0][0] == got[1][0] == 0.25
    assert got[0][1] == pytest.approx(2 * 545_891_164 / 0.25e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.5, None) == 1.5
    assert bench.whole_job_gbs(1_000_000_000, 1, 1.0) == pytest.approx(1000.0)
