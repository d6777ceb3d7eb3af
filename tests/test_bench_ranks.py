"""The multi-GPU bench path on the host: replicas only (no data-path collective),
the job time is the maximum over ranks and the value counts every replica's
work.  Run as two gloo ranks on CPU; the GPU work of each replica is the same
single-GPU step that the other tests cover."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")      # rank 1 is the slow one
        torch.distributed.barrier()
        out[rank] = ms
        # the reference arm runs on rank 0 only; the other ranks return without work
        if rank != 0:
            assert bench.run_reference(None, rank, world) is None
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_value(1_000_000, 1, 2.0)
    assert one == pytest.approx(500_000.0)                      # K-tokens/s
    assert bench.whole_job_value(1_000_000, 4, 2.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
