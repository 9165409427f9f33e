"""Host logic of the multi-GPU bench path (replicas, no data-path collective),
run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r "measured" 10 + r ms for its replica and 30 - r ms end to end
    total, e2e = bench.max_over_ranks([10.0 + rank, 30.0 - rank], dist, "cpu")
    results[rank] = (total, e2e, bench.job_throughput(1_000_000_000, world, 10, total))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank, args=(world, port, results), nprocs=world, start_method="spawn", join=True)
    assert results[0] == results[1]
    total, e2e, gbs = results[0]
    assert total == 11.0 and e2e == 30.0
    # 2 ranks x 10 steps x 1 GB over 11 ms
    assert gbs == pytest.approx(2 * 10 * 1.0 / 0.011)
