"""Host logic of the multi-GPU benchmark on CPU: world size 2, gloo.

The verify step shards over sequences with no exchange, so `bench.py --gpus N`
runs N replicas; the only cross-rank steps are the barrier and the max over
ranks of the timed region.  Here two CPU ranks check that reduction and the
whole-job rate built on it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [120.0, 150.0][rank]  # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, dist, "cpu")
    dist.barrier()
    out[rank] = (ms, bench.job_rate(2048, world, 10, ms))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 150.0
    assert rate == pytest.approx(2048 * 2 * 10 / 0.150)


def test_single_rank_passes_through():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_rate(2048, 1, 4000, 860.0) == pytest.approx(2048 * 4000 / 0.86)
