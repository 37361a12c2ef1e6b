"""GPU parity of the blockwise-scaled W8A8 GEMM (tcgen05) and its grouped MoE
variant against the float64 oracle: relative Frobenius error <= 1e-3 against
the BF16-rounded oracle and |dY| <= 4e-3 (|A| |W|^T) + 1e-6 per element, on
small cases spanning several tiles with ragged tails, on the full rollout
shapes with sampled outputs, and bit-exact on an exactly representable case."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, check_gemm, device, np_u8

pytestmark = pytest.mark.gpu


def _quantized(m, n, k, seed, dev):
    a = workloads.dense_acts(m, k, seed=seed, device=dev)
    w = workloads.make_weight(n, k, seed=seed + 1, device=dev)
    qa, sa = fp8rl.quantize_act_groupwise(a)
    qw, sw = fp8rl.quantize_weights_blockwise(w)
    return qa, sa, qw, sw


def _full_case(m, n, k, seed, ldy_pad=0):
    dev = device()
    qa, sa, qw, sw = _quantized(m, n, k, seed, dev)
    ldy = n + ldy_pad
    yc = Canary(m * ldy, torch.bfloat16, dev)
    y = yc.view.view(m, ldy)[:, :n]
    fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw, y)
    torch.cuda.synchronize()
    yc.check()
    if ldy_pad:
        pad = yc.view.view(m, ldy)[:, n:].contiguous().view(torch.uint8)
        assert (pad.cpu().numpy() == 0x5A).all(), "wrote into the row padding"
    y64, ab = oracle.gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw), sw.cpu().numpy())
    check_gemm(y, y64, ab, "m=%d n=%d k=%d" % (m, n, k))
    fp8rl.device_status(0)


def test_tiny_linear():
    dev = device()
    a, w = workloads.tiny_linear(seed=0)
    qa, sa = fp8rl.quantize_act_groupwise(a.to(dev))
    qw, sw = fp8rl.quantize_weights_blockwise(w.to(dev))
    y = fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw)
    y64, ab = oracle.gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw), sw.cpu().numpy())
    check_gemm(y, y64, ab, "tiny")
    fp8rl.device_status(0)


@pytest.mark.parametrize("m,n,k,ldy_pad", [(1, 256, 128, 0), (127, 512, 1024, 8), (129, 272, 256, 0),
                                           (300, 512, 384, 40), (64, 256, 512, 0),
                                           (513, 1024, 2048, 0), (200, 16, 128, 0),
                                           # wide flavour (128 x 256 tiles), several tiles
                                           # per CTA, ragged last n-tile; ragged last m-tile
                                           # (100 and 72 rows)
                                           (8192, 1392, 256, 8), (8292, 1392, 256, 0),
                                           (8264, 1280, 384, 16),
                                           # narrow flavour (128-wide tiles, four TMEM
                                           # buffers): ragged m and n tiles, padded rows
                                           (1500, 2576, 640, 8), (1300, 4096, 2048, 0),
                                           (1000, 1280, 640, 16),
                                           # split-K flavour (128-wide tiles): S = 3 with
                                           # uneven row slices and a ragged last m-tile,
                                           # no split possible (128 tiles: the narrow
                                           # flavour, one CTA per tile), S = 4 with a ragged
                                           # n-tile and padded rows, S = 2 (decode o)
                                           (200, 768, 384, 0), (500, 4096, 1024, 0),
                                           (100, 720, 4096, 24), (256, 4096, 1024, 0)])
def test_shapes(m, n, k, ldy_pad):
    _full_case(m, n, k, seed=m + n + k, ldy_pad=ldy_pad)


def test_exactly_representable_case_is_bit_exact():
    """Integer-valued codes (mostly zero), a power-of-two scale per row and per
    weight row-block that is the same for every k-block, and |sum| <= 256:
    every partial sum, every promotion and the BF16 result are exact, so the
    GPU must reproduce the oracle bit for bit."""
    dev = device()
    rng = np.random.default_rng(12)
    m, n, k = 200, 512, 512
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    small = np.array([c for c in range(0x7F) if float(table[c]).is_integer() and 0 < table[c] <= 2],
                     dtype=np.uint8)

    def codes(r, c):
        v = rng.choice(small, size=(r, c)) | (rng.integers(0, 2, (r, c)) << 7).astype(np.uint8)
        v[rng.random((r, c)) < 0.8] = 0
        return v.astype(np.uint8)

    qa, qw = codes(m, k), codes(n, k)
    sa = np.repeat(np.exp2(rng.integers(-4, -1, size=(1, m))), k // 128, axis=0).astype(np.float32)
    sw = np.repeat(np.exp2(rng.integers(-3, 0, size=(n // 128, 1))), k // 128, axis=1).astype(np.float32)
    y = fp8rl.gemm_w8a8_blockwise(torch.from_numpy(qa).to(dev), torch.from_numpy(sa).to(dev),
                                  torch.from_numpy(qw).to(dev), torch.from_numpy(sw).to(dev))
    y64, _ = oracle.gemm_w8a8(qa, sa, qw, sw)
    ref = oracle.bf16_round(y64)
    assert (ref.astype(np.float64) == y64).all()          # exact in bf16 by construction
    assert np.count_nonzero(y64) > y64.size // 2
    assert (y.float().cpu().numpy() == ref).all()


@pytest.mark.parametrize("m", [256, 8192])
def test_qwen3_8b_rollout_shapes_sampled(m):
    """act-quant + GEMM for qkv/o/gate_up/down at the decode and prefill
    token counts, checked on 48 sampled rows x 48 sampled columns each."""
    dev = device()
    rng = np.random.default_rng(m)
    for (name, n, k) in workloads.QWEN3_8B_LINEARS:
        qa, sa, qw, sw = _quantized(m, n, k, seed=workloads.sub_seed(3, m, n, k), dev=dev)
        y = fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw)
        torch.cuda.synchronize()
        rows = np.sort(rng.choice(m, size=48, replace=False))
        cols = np.sort(rng.choice(n, size=48, replace=False))
        rr = torch.from_numpy(rows).to(dev)
        cc = torch.from_numpy(cols).to(dev)
        qa_rows = np_u8(qa[rr])
        sa_rows = sa[:, rr].cpu().numpy()
        y64, ab = oracle.gemm_w8a8(qa_rows, np.ascontiguousarray(sa_rows), np_u8(qw),
                                   sw.cpu().numpy(), rows=None, cols=cols)
        check_gemm(y[rr][:, cc], y64, ab, "%s m=%d" % (name, m))
    fp8rl.device_status(0)


def _grouped_case(counts, n, k, seed, extra_rows=0):
    dev = device()
    E = len(counts)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    M = int(off[-1]) + extra_rows
    a = workloads.expert_inputs(M, k, seed=seed, device=dev)
    w = workloads.moe_weights(n, k, E, seed=seed + 1, device=dev)
    qa, sa = fp8rl.quantize_act_groupwise(a)
    qw2, sw2 = fp8rl.quantize_weights_blockwise(w.view(E * n, k))
    qw, sw = qw2.view(E, n, k), sw2.view(E, n // 128, k // 128)
    yc = Canary(M * n, torch.bfloat16, dev)
    y = yc.view.view(M, n)
    fp8rl.grouped_gemm_w8a8_blockwise(qa, sa, qw, sw, torch.from_numpy(off).to(dev), y)
    torch.cuda.synchronize()
    yc.check()
    return qa, sa, qw, sw, off, y, M


def test_grouped_small_with_empty_and_ragged_segments():
    counts = [3, 0, 130, 0, 7, 256, 1, 129]
    qa, sa, qw, sw, off, y, M = _grouped_case(counts, 256, 384, seed=21, extra_rows=5)
    y64, ab = oracle.grouped_gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw), sw.cpu().numpy(),
                                       off, rows=np.arange(int(off[-1])))
    check_gemm(y[:int(off[-1])], y64, ab, "grouped small")
    # rows beyond the last segment are never written
    tail = y[int(off[-1]):].contiguous().view(torch.uint8).cpu().numpy()
    assert (tail == 0x5A).all()
    fp8rl.device_status(0)


def _agree(y1, y2, absprod):
    """Two FP32-accumulated, BF16-rounded results of the same product that
    differ only in summation order: at most one BF16 ulp of the larger, plus
    FP32 reordering error on the scale of sum |a||w|."""
    a, b = y1.float().cpu().numpy(), y2.float().cpu().numpy()
    bound = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7 + absprod * 2.0 ** -16
    assert (np.abs(a - b) <= bound).all()


def test_grouped_single_expert_equals_dense():
    """One expert covering every row is the dense GEMM.  The dense call may
    split K across a cluster (few tiles), which changes only the FP32
    summation order: both meet the tolerance and differ by at most 1 BF16 ulp."""
    device()
    qa, sa, qw, sw, off, y, M = _grouped_case([300], 512, 256, seed=22)
    yd = fp8rl.gemm_w8a8_blockwise(qa, sa, qw[0].contiguous(), sw[0].contiguous())
    y64, ab = oracle.gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw[0]), sw[0].cpu().numpy())
    check_gemm(y, y64, ab, "grouped, one expert")
    check_gemm(yd, y64, ab, "dense")
    _agree(y, yd, ab)


def test_split_k_matches_unsplit_on_many_tiles():
    """The same product computed with few tiles (split-K cluster path) and as
    part of a larger launch (one CTA per tile): rows of the small problem must
    agree with the big one within 1 BF16 ulp, and both meet the tolerance."""
    dev = device()
    qa, sa, qw, sw = _quantized(1024, 2560, 1024, seed=23, dev=dev)
    y_big = fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw)                 # 8 x 10 wide tiles: no split
    qa_s = qa[:128].contiguous()
    sa_s = sa[:, :128].contiguous()
    y_small = fp8rl.gemm_w8a8_blockwise(qa_s, sa_s, qw, sw)           # 20 narrow tiles, S = 4
    y64, ab = oracle.gemm_w8a8(np_u8(qa_s), sa_s.cpu().numpy(), np_u8(qw), sw.cpu().numpy())
    check_gemm(y_small, y64, ab, "split-K")
    check_gemm(y_big[:128], y64, ab, "one CTA per tile")
    _agree(y_big[:128], y_small, ab)
    fp8rl.device_status(0)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_grouped_qwen3_30b_a3b_sampled(which):
    """128 experts, 4096 tokens routed top-8 with Zipf-skewed loads."""
    n, k = (2 * workloads.MOE_INTER, workloads.MOE_HIDDEN) if which == "gate_up" else \
        (workloads.MOE_HIDDEN, workloads.MOE_INTER)
    offsets, _, counts = workloads.moe_routing(seed=0)
    qa, sa, qw, sw, off, y, M = _grouped_case(counts.numpy(), n, k, seed=31)
    assert (off == offsets.numpy()).all()
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(M, size=96, replace=False))
    cols = np.sort(rng.choice(n, size=32, replace=False))
    y64, ab = oracle.grouped_gemm_w8a8(np_u8(qa), sa.cpu().numpy(), np_u8(qw), sw.cpu().numpy(),
                                       off, rows=rows, cols=cols)
    dev = y.device
    check_gemm(y[torch.from_numpy(rows).to(dev)][:, torch.from_numpy(cols).to(dev)], y64, ab,
               "moe " + which)
    fp8rl.device_status(0)
