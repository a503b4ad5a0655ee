"""The multi-GPU path of bench.py is replicas only (the layer has no cross-token exchange):
each rank runs the whole workload on its own GPU and the job time is the slowest rank's.
This checks that host logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [12.5, 20.0][rank]  # ms: rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed)
    out[rank] = (mx, bench.replica_throughput(64, 10, world, mx))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        mx, tput = out[rank]
        assert mx == 20.0
        assert tput == pytest.approx(2 * 64 * 10 / 0.020)


def test_single_process_is_a_noop():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.replica_throughput(32, 5, 1, 10.0) == pytest.approx(32 * 5 / 0.010)
