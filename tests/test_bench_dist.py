"""Host logic of the multi-process bench (replicas, no data-path collective):
max-over-ranks timing and whole-job aggregation across two gloo ranks on CPU,
and the reference arm's behaviour on ranks other than 0."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench._dist()
        # rank r "took" (10 + 5 r) ms in total and (4 + r) ms in the re-quant row
        total, a1 = bench.max_over_ranks([10.0 + 5 * r, 4.0 + r], torch.device("cpu"), w)
        value = bench.replica_gbs(w, 1e9, 3, a1)
        q.put((r, w, local, total, a1, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_over_ranks_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, local, total, a1, value in out:
        assert w == 2 and local == r
        assert total == 15.0 and a1 == 5.0          # the slowest rank's times on every rank
        assert value == pytest.approx(2 * 1e9 * 3 / 5e-3 / 1e9)   # 2 replicas / slowest time


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.0, 7.5], torch.device("cpu"), 1) == [3.0, 7.5]
    assert bench.replica_gbs(1, 2e9, 4, 1000.0) == pytest.approx(8.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"gpus": 2, "steps": 1, "warmup": 3})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(args)
    assert rc == 0 and buf.getvalue() == ""
