"""The N > 1 path of bench.py on CPU: two gloo ranks with different step times agree on
the slowest one, and the whole-job rate counts every rank's units (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [0.001 * (rank + 1), 0.010 + 0.002 * rank]      # fwd, decode seconds
    fwd, dec = bench.max_over_ranks(times, world, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 16384, fwd)
    out.put((rank, fwd, dec, rate))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_rate_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, fwd, dec, rate in res:
        assert fwd == pytest.approx(0.001 * world)
        assert dec == pytest.approx(0.010 + 0.002 * (world - 1))
        assert rate == pytest.approx(world * 16384 / (0.001 * world))


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]
    assert bench.whole_job_rate(1, 100, 2.0) == 50.0
