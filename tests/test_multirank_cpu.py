"""bench.py's multi-rank host logic on CPU: two gloo ranks, each a replica of the
workload, agree on the slowest rank's time and report the whole-job value."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [40.0, 55.0][rank]
    m = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    bench.barrier(world)
    out[rank] = (m, bench.job_value(1e12, world, m))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 55.0
    # two replicas of 1e12 flops each in 55 ms
    assert res[0][1] == pytest.approx(2e12 / 0.055 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_value(3.518e13, 1, 30.0) == pytest.approx(1172.67, rel=1e-4)


def test_host_buffer_placement_helpers():
    """The e2e buffers' placement: CPU lists print compactly, and without a GPU (or its
    sysfs entry) the placement leaves the process's CPU set untouched."""
    import bench
    assert bench.cpu_list({0, 1, 2, 3, 5, 7, 8, 9}) == "0-3,5,7-9"
    assert bench.cpu_list({4}) == "4"
    before = os.sched_getaffinity(0)
    with bench.near_gpu(torch.device("cpu")) as cpus:
        assert cpus is None
        assert os.sched_getaffinity(0) == before
    assert os.sched_getaffinity(0) == before
