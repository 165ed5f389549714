"""The N > 1 benchmark path on the CPU: two gloo ranks, each timing its own replica
(the forward has no exchange step). The reported time is the maximum over ranks and
the value counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = [10.0, 12.5][rank]
    mx = bench.reduce_over_ranks(my_ms, world, torch.device("cpu"))
    val = bench.aggregate_value(1e12, 100, world, mx)
    out[rank] = (mx, val)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        mx, val = out[r]
        assert mx == pytest.approx(12.5)
        # 2 ranks x 100 steps x 1 TFLOP in 12.5 ms
        assert val == pytest.approx(2 * 100 * 1.0 / 12.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 1) == 3.0
    assert bench.aggregate_value(2e12, 10, 1, 20.0) == pytest.approx(1000.0)
