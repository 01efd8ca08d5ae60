"""The N > 1 bench path on CPU: two gloo ranks, each a replica of the workload.

The product needs no exchange, so the only cross-rank logic is the timing
aggregation: the slowest rank's time over the whole job's work."""
import os

import pytest
import torch.multiprocessing as mp


def _rank_main(rank, world, port, out):
    import torch.distributed as tdist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0 + rank, 3.0 - rank]                 # rank 0: (2, 3); rank 1: (3, 2)
        got = bench.max_over_ranks(ms, "cpu")
        out[rank] = (got, bench.whole_job_tflops(world, 1e12, got[0]))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for rank in (0, 1):
        got, tflops = out[rank]
        assert got == [3.0, 3.0]
        assert tflops == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.whole_job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
