"""GPU parity of the decode-sized linear layer (activation quantization fused
with the W8A8 GEMM, stream-K over every SM) against the oracle: the codes and
scales bit for bit, Y within the GEMM tolerances; on the Qwen3-8B decode
shapes (M = 256) and ragged ones, with tile splits over 1, 2, 3 and more
CTAs, the GEMM-only mode, repeated calls on one workspace, and a graph
replay."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, check_gemm, device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _segments_per_tile(n, k, sms):
    """Host copy of the stream-K deal: how many CTAs share each output tile."""
    tiles, kb = n // 128, k // 128
    U = tiles * kb
    grid = min(sms, U)
    owner = lambda x: ((x + 1) * grid - 1) // U    # noqa: E731
    return [owner(t * kb + kb - 1) - owner(t * kb) + 1 for t in range(tiles)]


def _case(dev, m, n, k, seed, rows=None, cols=None, workspace=None, fused=True):
    a = workloads.dense_acts(m, k, seed=seed)
    w = workloads.make_weight(n, k, seed=seed + 1)
    qw, sw = fp8rl.quantize_weights_blockwise(w.to(dev))
    yc = Canary(m * n, torch.bfloat16, dev)
    if fused:
        y, qa, sa = fp8rl.linear_w8a8_decode(a.to(dev), qw, sw, y=yc.view.view(m, n),
                                             workspace=workspace)
    else:
        qa, sa = fp8rl.quantize_act_groupwise(a.to(dev))
        y, _, _ = fp8rl.linear_w8a8_decode(None, qw, sw, y=yc.view.view(m, n), qa=qa, sa=sa,
                                           workspace=workspace)
    torch.cuda.synchronize()
    yc.check()
    fp8rl.device_status(0)
    oqa, osa = oracle.quantize_act_groupwise(a)
    assert (np_u8(qa) == oqa).all(), "codes"
    assert (np_f32_bits(sa) == osa.view(np.uint32)).all(), "scales"
    r = np.arange(m) if rows is None else rows
    c = np.arange(n) if cols is None else cols
    y64, ab = oracle.gemm_w8a8(oqa, osa, np_u8(qw), sw.cpu().numpy(), rows=r, cols=c)
    check_gemm(y[torch.from_numpy(r).to(dev)][:, torch.from_numpy(c).to(dev)], y64, ab,
               "decode m=%d n=%d k=%d" % (m, n, k))
    return y


@pytest.mark.parametrize("name,n,k", [("qkv", 6144, 4096), ("o", 4096, 4096),
                                      ("gate_up", 24576, 4096), ("down", 4096, 12288)])
def test_qwen3_8b_decode_shapes(name, n, k):
    dev = device()
    rng = np.random.default_rng(n + k)
    _case(dev, 256, n, k, seed=50 + n % 97, rows=np.sort(rng.choice(256, 48, replace=False)),
          cols=np.sort(rng.choice(n, 96, replace=False)))


@pytest.mark.parametrize("m,n,k", [(1, 128, 128), (17, 384, 640), (100, 1280, 4096),
                                   (255, 2048, 1024), (256, 512, 256), (64, 19456, 1024)])
def test_ragged_shapes(m, n, k):
    dev = device()
    _case(dev, m, n, k, seed=m + n + k)


def test_tile_splits_over_one_to_many_ctas():
    dev = device()
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    seen = set()
    for n, k in ((128 * grid, 1024), (24576, 4096), (12288, 2048), (6144, 1536), (1280, 4096)):
        seen.update(_segments_per_tile(n, k, grid))
        rng = np.random.default_rng(n)
        _case(dev, 256, n, k, seed=n % 1000, rows=np.sort(rng.choice(256, 40, replace=False)),
              cols=np.sort(rng.choice(n, 80, replace=False)))
    assert {1, 2, 3} <= seen and max(seen) > 8


def test_gemm_only_mode_and_repeated_calls_on_one_workspace():
    dev = device()
    n, k, m = 4096, 2048, 200
    ws = torch.zeros(fp8rl.linear_w8a8_decode_workspace_bytes(n), dtype=torch.uint8, device=dev)
    y1 = _case(dev, m, n, k, seed=7, workspace=ws, fused=False)
    y2 = _case(dev, m, n, k, seed=7, workspace=ws)
    y3 = _case(dev, m, n, k, seed=7, workspace=ws)
    assert torch.equal(y2.view(torch.int16), y3.view(torch.int16))      # deterministic
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))      # same A codes and scales


def test_agrees_with_the_dense_gemm():
    """Same codes and scales through the dense kernel: the two differ only in
    the FP32 order of the partial sums, so they agree within twice the
    per-element GEMM bound (each is within it of the float64 result)."""
    dev = device()
    a = workloads.dense_acts(256, 4096, seed=9).to(dev)
    qw, sw = fp8rl.quantize_weights_blockwise(workloads.make_weight(6144, 4096, seed=10).to(dev))
    y, qa, sa = fp8rl.linear_w8a8_decode(a, qw, sw)
    yd = fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw)
    torch.cuda.synchronize()
    rows = np.arange(0, 256, 5)
    _, ab = oracle.gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw), sw.cpu().numpy(), rows=rows)
    d = (y.float() - yd.float()).abs().cpu().numpy().astype(np.float64)[rows]
    assert (d <= 2 * (4e-3 * ab + 1e-6)).all()
    assert (d == 0).mean() > 0.5      # most outputs are bit-identical


def test_graph_replay():
    dev = device()
    a = workloads.dense_acts(256, 4096, seed=11).to(dev)
    qw, sw = fp8rl.quantize_weights_blockwise(workloads.make_weight(4096, 4096, seed=12).to(dev))
    ws = torch.zeros(fp8rl.linear_w8a8_decode_workspace_bytes(4096), dtype=torch.uint8, device=dev)
    y_e, qa_e, sa_e = fp8rl.linear_w8a8_decode(a, qw, sw, workspace=ws)
    torch.cuda.synchronize()
    y = torch.zeros_like(y_e)
    qa = torch.zeros_like(qa_e)
    sa = torch.zeros_like(sa_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fp8rl.linear_w8a8_decode(a, qw, sw, y=y, qa=qa, sa=sa, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp8rl.linear_w8a8_decode(a, qw, sw, y=y, qa=qa, sa=sa, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    assert torch.equal(y.view(torch.int16), y_e.view(torch.int16))
    assert torch.equal(qa, qa_e) and torch.equal(sa.view(torch.int32), sa_e.view(torch.int32))
