"""The N > 1 host path of bench.py (replicas: one process per GPU, no data
exchange) on CPU ranks with gloo: the barrier, the max over ranks of the
timings, and the whole-job throughput built from it."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(w, 10.0 + rank)          # rank r "took" 10 + r ms
    out[rank] = t
    out[world + rank] = bench.aggregate_gbs(w, 1e9, 4, t)
    bench.barrier(w)
    torch.distributed.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the host-only one")
def test_two_replicas_share_the_slowest_time():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * (2 * world))
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert list(out[:world]) == [11.0, 11.0]            # both ranks see the max
    # 2 replicas x 1 GB x 4 steps over 11 ms
    assert out[world] == out[world + 1] == pytest.approx(2 * 1e9 * 4 / 11e-3 / 1e9)


def test_single_process_passes_through():
    import bench
    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.aggregate_gbs(1, 2e9, 10, 5.0) == pytest.approx(4000.0)
