"""The multi-GPU form of the bench is N independent replicas (the path has no
data exchange on one GPU per rank): each rank times its own step and the job
reports all ranks' tokens over the slowest rank's time. This checks that
host-side logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        ms = bench.max_over_ranks(times[rank], w, device="cpu")
        out.put((r, ms, bench.whole_job_tokens_per_s(8192, w, ms)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(13.0, 13.5), (20.0, 10.0)])
def test_two_replicas_report_the_slowest(times):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in procs)
    slow = max(times)
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, value in res:
        assert ms == slow
        assert abs(value - 2 * 8192 / (slow / 1e3)) < 1e-6 * value


def test_one_rank_is_its_own_time():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_tokens_per_s(8192, 1, 12.5) == 8192 / 0.0125
