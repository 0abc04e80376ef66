"""Multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.  The forward
shards over independent (sequence, head) units with no data-path exchange, so the only
cross-rank step is the timing aggregation: the step time is the maximum over ranks and the
work is the sum over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, units, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        t, u = bench.aggregate(times[rank], units[rank], world)
        out[rank] = (t, u)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_aggregate_max_time_sum_units(world):
    times = [0.125, 0.5]
    units = [1_048_576, 524_288]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, units, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        t, u = res[r]
        assert t == max(times)
        assert u == float(sum(units))


def test_aggregate_single_rank_is_identity():
    import bench

    assert bench.aggregate(0.25, 123, 1) == (0.25, 123)
