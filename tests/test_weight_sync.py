"""Sharded quantize-then-all-gather weight sync (summary page, section 3.4.2
Phase 2), host side: the shard plan (whole 128-row block bands, contiguous,
balanced, covering every row), and the gather itself on world-size 2 and 3
gloo groups on CPU.  On CPU the ranks quantize their shards with the oracle
(passed in as the quantizer; the library's kernel needs a GPU): the gathered
codes and scales must equal the oracle's quantization of every whole tensor
bit for bit, which checks the plan, the packing, the padding of uneven
pieces and the reassembly."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import __graft_entry__
from fp8_precision_rollout_gb300 import binding, weight_sync, workloads

SHAPES = [(1000, 264), (128, 136), (7, 8), (640, 1024), (300, 512)]


def _lib():
    __graft_entry__.build()
    return binding.load()


def test_shard_plan_covers_rows_in_whole_bands():
    _lib()
    for n in (0, 1, 7, 127, 128, 129, 1000, 4096, 24576, 24577):
        for world in (1, 2, 3, 4, 7, 8, 64):
            rows = [binding.weight_shard_rows(n, world, r) for r in range(world)]
            assert rows[0][0] == 0 and rows[-1][1] == n
            for (b0, e0), (b1, e1) in zip(rows, rows[1:]):
                assert e0 == b1                              # contiguous, in rank order
            for b, e in rows:
                assert b % 128 == 0 and (e % 128 == 0 or e == n) and b <= e
            bands = [(e - b + 127) // 128 for b, e in rows]
            assert max(bands) - min(bands) <= 1             # balanced


def test_shard_plan_rejects_bad_arguments():
    L = _lib()
    import ctypes
    b, e = ctypes.c_int64(), ctypes.c_int64()
    assert L.fp8rl_weight_shard_rows(10, 2, 2, ctypes.byref(b), ctypes.byref(e)) == 1
    assert L.fp8rl_weight_shard_rows(-1, 2, 0, ctypes.byref(b), ctypes.byref(e)) == 1
    assert L.fp8rl_weight_shard_rows(10, 0, 0, ctypes.byref(b), ctypes.byref(e)) == 1


def test_fp8_gather_moves_about_half_the_bf16_bytes():
    _lib()
    g = weight_sync.gathered_bytes([(6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288)], 8)
    assert g["fp8_codes_and_scales"] < 0.51 * g["bf16"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_quantize(shards):
    import oracle
    qs, ss = [], []
    for w in shards:
        if w.shape[0] == 0:
            qs.append(torch.empty(0, w.shape[1], dtype=torch.uint8))
            ss.append(torch.empty(0, (w.shape[1] + 127) // 128, dtype=torch.float32))
            continue
        q, s = oracle.quantize_weights_blockwise(w)
        qs.append(torch.from_numpy(q))
        ss.append(torch.from_numpy(s))
    return qs, ss


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        full = [workloads.make_weight(n, k, seed=300 + i) for i, (n, k) in enumerate(SHAPES)]
        rows = weight_sync.plan(SHAPES, world)[rank]
        shards = [w[b:e].contiguous() for w, (b, e) in zip(full, rows)]
        gq, gs = weight_sync.sync_weights(shards, SHAPES, quantize=_oracle_quantize)
        q.put((rank, [x.numpy() for x in gq], [x.numpy() for x in gs]))
    finally:
        dist.destroy_process_group()


def _run(world):
    import oracle
    _lib()
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = [workloads.make_weight(n, k, seed=300 + i) for i, (n, k) in enumerate(SHAPES)]
    want = [oracle.quantize_weights_blockwise(w) for w in full]
    for rank, gq, gs in out:
        for i, (wq, ws_) in enumerate(want):
            assert (gq[i] == wq).all(), (rank, i)
            assert (gs[i].view(np.uint32) == ws_.view(np.uint32)).all(), (rank, i)


def test_gather_two_ranks():
    _run(2)


def test_gather_three_ranks_with_an_empty_shard():
    # the (7, 8) and (128, 136) tensors have one row band: two of three ranks own none
    _run(3)
