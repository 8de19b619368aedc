"""The multi-GPU form of the benchmark: independent replicas, one per rank, with
the job timed by its slowest rank.  Checked on CPU with the gloo backend and
two ranks (no GPU is involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [1.5, 4.0][rank]  # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        results[rank] = (ms, bench.job_value(1_000_000, world, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), results), nprocs=2, join=True,
                           start_method="spawn")
        got = dict(results)
    assert got[0][0] == got[1][0] == 4.0
    # 2 ranks x 1e6 elements in 4 ms = 0.5 Gelem/s on every rank
    assert abs(got[0][1] - 0.5) < 1e-12 and got[0][1] == got[1][1]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert abs(bench.job_value(2_000_000, 1, 2.0) - 1.0) < 1e-12
