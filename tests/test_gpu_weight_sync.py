"""The sharded weight sync's quantization on the GPU: every rank's shards
quantized by the library's multi-tensor kernel, packed as the all-gather
sends them and reassembled, equal the whole tensors' codes and scales bit for
bit (the library's and the oracle's).  The ranks run one after another on one
GPU: each rank's work is independent and only the exchange is collective
(tested with gloo ranks on CPU in test_weight_sync.py)."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import weight_sync, workloads
from gpu_helpers import device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _simulate(shapes, full, world, dev):
    plans = weight_sync.plan(shapes, world)
    sizes = [weight_sync._piece_sizes(shapes, p) for p in plans]
    q_len = max(1, max(s[0] for s in sizes))
    s_len = max(1, max(s[1] for s in sizes))
    qp, sp = [], []
    for r in range(world):
        shards = [w[b:e].contiguous() for w, (b, e) in zip(full, plans[r])]
        qs, ss = weight_sync.quantize_local(shards)
        q, s = weight_sync.pack_piece(qs, ss, q_len, s_len, dev)
        qp.append(q)
        sp.append(s)
    return weight_sync.assemble(shapes, plans, qp, sp)


@pytest.mark.parametrize("world", [2, 3, 8])
def test_ragged_tensors(world):
    dev = device()
    shapes = [(1000, 264), (128, 136), (7, 8), (640, 1024), (300, 512), (2049, 256)]
    full = [workloads.make_weight(n, k, seed=400 + i, device=dev) for i, (n, k) in enumerate(shapes)]
    gq, gs = _simulate(shapes, full, world, dev)
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    for i, w in enumerate(full):
        oq, os_ = oracle.quantize_weights_blockwise(w.cpu())
        assert (np_u8(gq[i]) == oq).all(), i
        assert (np_f32_bits(gs[i]) == os_.view(np.uint32)).all(), i


def test_qwen3_8b_layer0_over_8_ranks():
    dev = device()
    shapes = [(n, k) for _, n, k in workloads.QWEN3_8B_LINEARS]
    full = [workloads.make_weight(n, k, seed=workloads.sub_seed(2, 0, i), device=dev)
            for i, (n, k) in enumerate(shapes)]
    gq, gs = _simulate(shapes, full, 8, dev)
    fq, fs = fp8rl.quantize_weights_blockwise_multi(full)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(gq[i], fq[i]) and torch.equal(gs[i].view(torch.int32),
                                                         fs[i].view(torch.int32))
    oq, os_ = oracle.quantize_weights_blockwise(full[0].cpu())
    assert (np_u8(gq[0]) == oq).all() and (np_f32_bits(gs[0]) == os_.view(np.uint32)).all()
