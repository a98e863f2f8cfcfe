"""The bench's multi-GPU path is replicas only (independent copies of the decode path, no data-path
collective): the host side that joins them — the maximum of each timing over the ranks and the
whole-job rate — run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's decode, prefill and end-to-end seconds
        mine = [1.0 + rank, 0.5 - 0.25 * rank, 2.0 + 0.5 * rank]
        out[rank] = bench.max_over_ranks(mine, world)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks_and_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(out)
    assert got[0] == got[1] == [2.0, 0.5, 2.5]
    # 2 replicas x 20 steps of one token in the slowest replica's 2.0 s
    assert bench.job_rate(20, world, got[0][0]) == pytest.approx(20.0)


def test_single_process_keeps_its_own_times():
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_rate(256, 1, 2.0) == 128.0
