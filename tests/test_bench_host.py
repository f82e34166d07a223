"""Host logic of bench.py without a GPU: the whole-job aggregation over ranks
(max of elapsed time, sum of work) on a world_size-2 gloo group, and the clock
sampler's parsing of nvidia-smi CSV."""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed, units = bench.aggregate(dist, elapsed_s=1.0 + rank, units=10.0 * (rank + 1))
    out[rank] = (elapsed, units)
    dist.destroy_process_group()


def test_aggregate_is_max_time_and_sum_of_work_over_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (2.0, 30.0)


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate(None, 1.5, 7.0) == (1.5, 7.0)


def test_clock_sampler_parses_throttle_reasons(tmp_path):
    import bench
    s = bench.ClockSampler(0)
    f = tmp_path / "c.csv"
    f.write_text("0, 1980, 2070, 700.5, 0x0, Not Active, Not Active, Not Active, Active\n"
                 "0, 2000, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Not Active\n")
    s.file = open(f, "a+")
    s.proc = object()
    summ = s.summary()
    assert summ["sm_mhz"] == 1990.0 and summ["sm_max_mhz"] == 2070.0
    assert summ["reasons"] == ["sw_power_cap"] and summ["samples"] == 2
