"""Host logic of the benchmark: algorithmic byte counts, the replica launch
(two gloo ranks on the CPU through torch.distributed.run), per-rank seeds and
the max-over-ranks step time."""
import json
import os
import socket
import subprocess
import sys

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


def test_algorithmic_bytes_sweep_and_stack():
    """Per-step bytes of the sweep (gamma = 4 column) and the 8-layer stack."""
    MB = 1e6
    lo = bench.algorithmic_bytes(WORKLOADS["sweep32k"].with_(k=512, gamma=4, m=128))
    hi = bench.algorithmic_bytes(WORKLOADS["sweep32k"].with_(k=4096, gamma=4, m=1024))
    assert lo["score"] / MB == pytest.approx(337.6, abs=0.1)
    assert lo["step"] / MB == pytest.approx(358.7, abs=0.2)
    assert hi["step"] / MB == pytest.approx(476.3, abs=0.2)
    assert lo["dense"] / MB == pytest.approx(1075.9, abs=0.5)
    st = bench.algorithmic_bytes(WORKLOADS["stack128k"])
    assert st["score"] / MB == pytest.approx(675.3, abs=0.1)
    assert st["verify"] / MB == pytest.approx(545.5, abs=0.2)
    assert st["step"] / MB == pytest.approx(1225.0, abs=0.3)
    # 3 rows of K and V, read from the block and written to the cache, 8 layers
    assert bench.append_bytes(WORKLOADS["stack128k"], 3) == 8 * 2 * 2 * 4 * 8 * 3 * 128 * 2 + 32


def test_replica_launch_two_gloo_ranks():
    """--gpus N without a torchrun environment starts N ranks through
    torch.distributed.run; each rank gets its own seed and the step time is
    the max over ranks (gloo here, NCCL with GPUs)."""
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_replica_probe.py")
    cmd = bench.replica_command(2, [], script=probe)
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=2" in cmd
    assert "127.0.0.1" in cmd
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(v, None)
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert out["world"] == 2 and out["backend"] == "gloo"
    assert len(set(out["seeds"])) == 2
    assert out["max"] == 2.0


def test_gpus_must_match_world_size():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"),
                        "--gpus", "2"], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 2 and "WORLD_SIZE=1" in r.stderr


def test_cpu_model_string():
    name = bench.cpu_model()
    assert isinstance(name, str) and name and name not in ("aarch64",)
