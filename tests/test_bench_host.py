"""Host logic of the multi-replica benchmark, on CPU with gloo (world size 2).

The benchmark runs one independent replica of the decode step per GPU; the
only cross-rank steps are a barrier around the timed region and the maximum
of the ranks' times, from which the whole-job throughput is computed.  These
tests run that logic in two CPU processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, local = bench.dist_init("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    mx = bench.max_over_ranks(times[rank], w, device="cpu")
    out[rank] = (mx, bench.job_throughput(1e9, mx, w))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_two_ranks():
    world = 2
    times = [1.5, 2.0]          # ms per step on rank 0 and rank 1
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        mx, gbs = res[r]
        assert mx == 2.0                       # every rank sees the slowest time
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)   # both replicas' bytes / slowest time


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(2e9, 1.0, 1) == pytest.approx(2000.0)
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_init()[0] == 1
