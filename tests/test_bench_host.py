"""Host logic of the benchmark: algorithmic byte counts and the max-over-ranks
step time with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from synth import WORKLOADS


def test_algorithmic_bytes_headline():
    ab = bench.algorithmic_bytes(WORKLOADS["batched32k"])
    MB = 1e6
    assert ab["score"] / MB == pytest.approx(675.3, abs=0.1)
    assert ab["select"] / MB == pytest.approx(4.3, abs=0.1)
    assert ab["verify"] / MB == pytest.approx(139.5, abs=0.1)
    assert ab["step"] / MB == pytest.approx(819.1, abs=0.2)
    assert ab["dense"] / MB == pytest.approx(2152.6, abs=0.5)
    assert len(bench.slabs(WORKLOADS["batched32k"])) == 6


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_single_rank_passthrough():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
