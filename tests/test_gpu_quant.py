"""GPU parity of the quantizers against the CPU oracle: bit-exact codes and
scales on the same seeded inputs, ragged shapes, special values, an
exhaustive sweep of the element map over every BF16 (x, amax) pair, and the
full-size Qwen3-8B re-quantization and long-context KV workloads on sampled
blocks / rows."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _act_case(a_cpu, dev, lda_pad=0):
    m, k = a_cpu.shape
    if lda_pad:
        big = torch.zeros(m, k + lda_pad, dtype=torch.bfloat16, device=dev)
        big[:, :k] = a_cpu.to(dev)
        a = big[:, :k]
    else:
        a = a_cpu.to(dev)
    qc = Canary(m * k, torch.uint8, dev)
    sc = Canary(((k + 127) // 128) * m, torch.float32, dev)
    q, s = fp8rl.quantize_act_groupwise(a, qc.view.view(m, k), sc.view.view((k + 127) // 128, m))
    torch.cuda.synchronize()
    qc.check(); sc.check()
    oq, os_ = oracle.quantize_act_groupwise(a_cpu)
    assert (np_u8(q) == oq).all()
    assert (np_f32_bits(s) == os_.view(np.uint32)).all()


@pytest.mark.parametrize("m,k", [(64, 512), (1, 8), (3, 200), (127, 1032), (129, 4104), (70, 768),
                                 (300, 4096), (256, 12288), (5, 1024 + 24)])
def test_act_quant_shapes(m, k):
    dev = device()
    _act_case(workloads.dense_acts(m, k, seed=m * 7 + k), dev)


def test_act_quant_row_stride():
    dev = device()
    _act_case(workloads.dense_acts(33, 640, seed=3), dev, lda_pad=136)


def test_act_quant_tiny_linear_outlier_columns():
    dev = device()
    a, _ = workloads.tiny_linear(seed=0)
    _act_case(a, dev)


def test_act_quant_special_values():
    dev = device()
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=(40, 1024)).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF          # no inf/NaN (out of contract)
    bits[0] = 0                                         # all-zero row -> scale 0
    bits[1] = 0x8000                                    # all -0
    bits[2, :] = 0x0001                                 # smallest subnormals
    bits[3, ::2] = 0x7F7F                               # bf16 max
    bits[4, :] = rng.integers(0, 0x80, size=1024)       # subnormals only
    bits[5, :128] = 0x3F80                              # exactly 1.0 (amax 1)
    a = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    _act_case(a, dev)


@pytest.mark.parametrize("m", [256, 8192])
def test_act_quant_rollout_shapes_full(m):
    dev = device()
    for k in (4096, 12288):
        _act_case(workloads.dense_acts(m, k, seed=m + k), dev)


def test_element_map_exhaustive_over_bf16_pairs():
    """Every BF16 amax (positive finite) against every BF16 x with |x| <= amax,
    both signs: each 1x128 group holds amax followed by 127 x values."""
    dev = device()
    amaxes = np.arange(1, 0x7F80, dtype=np.int64)
    chunk = 1024
    for c0 in range(0, amaxes.size, chunk):
        am = amaxes[c0:c0 + chunk]
        counts = 2 * (am + 1)                          # x in [0, amax] and [-0, -amax]
        groups = (counts + 126) // 127
        total = int(groups.sum())
        rows = np.zeros((total, 128), dtype=np.uint16)
        gstart = np.concatenate([[0], np.cumsum(groups)])
        for i, a in enumerate(am):
            vals = np.arange(0, a + 1, dtype=np.uint16)
            vals = np.concatenate([vals, vals | 0x8000])
            g0, g1 = gstart[i], gstart[i + 1]
            blk = np.zeros(((g1 - g0) * 127,), dtype=np.uint16)
            blk[:vals.size] = vals
            rows[g0:g1, 0] = a
            rows[g0:g1, 1:] = blk.reshape(-1, 127)
        a_cpu = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)
        q, s = fp8rl.quantize_act_groupwise(a_cpu.to(dev))
        oq, os_ = oracle.quantize_act_groupwise(a_cpu)
        assert (np_f32_bits(s) == os_.view(np.uint32)).all(), "scales, amax chunk %d" % c0
        bad = np_u8(q) != oq
        assert not bad.any(), "codes differ at %s" % (np.argwhere(bad)[:5],)


def _wq_case(w_cpu, dev, ldw_pad=0, ldq_pad=0):
    n, k = w_cpu.shape
    if ldw_pad:
        big = torch.zeros(n, k + ldw_pad, dtype=torch.bfloat16, device=dev)
        big[:, :k] = w_cpu.to(dev)
        w = big[:, :k]
    else:
        w = w_cpu.to(dev)
    ldq = k + ldq_pad
    qc = Canary(n * ldq, torch.uint8, dev)
    qv = qc.view.view(n, ldq)[:, :k]
    nb, kb = (n + 127) // 128, (k + 127) // 128
    sc = Canary(nb * kb, torch.float32, dev)
    fp8rl.quantize_weights_blockwise(w, qv, sc.view.view(nb, kb))
    torch.cuda.synchronize()
    qc.check(); sc.check()
    oq, os_ = oracle.quantize_weights_blockwise(w_cpu)
    assert (np_u8(qv) == oq).all()
    assert (np_f32_bits(sc.view) == os_.reshape(-1).view(np.uint32)).all()
    if ldq_pad:   # padding columns of q are untouched
        assert (np_u8(qc.view.view(n, ldq)[:, k:]) == 0x5A).all()


@pytest.mark.parametrize("n,k", [(256, 512), (130, 200), (1, 8), (257, 1000), (6144, 4096),
                                 (128, 128), (4096, 12288)])
def test_weight_quant_shapes(n, k):
    dev = device()
    _wq_case(workloads.make_weight(n, k, seed=n + 3 * k), dev)


def test_weight_quant_special_values():
    """One pattern per 128x128 block: zeros of both signs (scale 0), the
    smallest subnormals, BF16 max, subnormals only, exactly 1.0, values near
    1e-20 (a scale below 2^-60: the IEEE-division branch), one outlier among
    tiny values; random finite bit patterns elsewhere; then a ragged copy."""
    dev = device()
    rng = np.random.default_rng(17)
    bits = rng.integers(0, 1 << 16, size=(384, 512)).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF          # no inf/NaN (out of contract)
    blk = lambda i, j: (slice(128 * i, 128 * i + 128), slice(128 * j, 128 * j + 128))  # noqa: E731
    bits[blk(0, 0)] = 0
    bits[blk(0, 1)] = 0x8000
    bits[blk(0, 2)] = 0x0001
    b = bits[blk(0, 3)]; b[::3, ::5] = 0x7F7F; b[1::3, ::5] = 0xFF7F
    bits[blk(1, 0)] = rng.integers(0, 0x80, size=(128, 128)) | (rng.integers(0, 2, size=(128, 128)) << 15)
    bits[blk(1, 1)] = 0x3F80
    tiny = (rng.normal(0, 1, size=(128, 128)) * 1e-20).astype(np.float32)
    bits[blk(1, 2)] = (tiny.view(np.uint32) >> 16).astype(np.uint16)
    small = (rng.normal(0, 1, size=(128, 128)) * 1e-3).astype(np.float32)
    small[77, 3] = -250.0
    bits[blk(1, 3)] = (small.view(np.uint32) >> 16).astype(np.uint16)
    w = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    _wq_case(w, dev)
    _wq_case(w[:300, :520].contiguous(), dev)


def test_weight_quant_strides():
    dev = device()
    _wq_case(workloads.make_weight(300, 520, seed=9), dev, ldw_pad=40, ldq_pad=24)


def test_weight_quant_multi_batches_and_chunking():
    dev = device()
    shapes = [(256, 512), (130, 200), (1, 8), (640, 1024), (128, 136), (3, 4096), (129, 129 + 7)]
    shapes = [(n, k - k % 8) for n, k in shapes]
    ws = [workloads.make_weight(n, k, seed=i) for i, (n, k) in enumerate(shapes)]
    # more tensors than one launch takes (160 descriptors per launch)
    ws += [workloads.make_weight(8, 16, seed=1000 + i) for i in range(300)]
    qs, ss = fp8rl.quantize_weights_blockwise_multi([w.to(dev) for w in ws])
    torch.cuda.synchronize()
    for w, q, s in zip(ws, qs, ss):
        oq, os_ = oracle.quantize_weights_blockwise(w)
        assert (np_u8(q) == oq).all()
        assert (np_f32_bits(s) == os_.view(np.uint32)).all()


def test_requant_qwen3_8b_full_model_sampled():
    """The whole Qwen3-8B linear stack (36 x 4 tensors, 6.95 G elements) in one
    multi-tensor call, checked on sampled blocks of every tensor."""
    dev = device()
    rng = np.random.default_rng(0)
    shapes = workloads.qwen3_8b_linear_shapes()
    ws = [workloads.make_weight(n, k, seed=workloads.sub_seed(2, l, i), device=dev)
          for i, (l, _, n, k) in enumerate(shapes)]
    qs, ss = fp8rl.quantize_weights_blockwise_multi(ws)
    torch.cuda.synchronize()
    for w, q, s in zip(ws, qs, ss):
        n, k = w.shape
        nb, kb = n // 128, k // 128
        ids = rng.choice(nb * kb, size=4, replace=False)
        for b in ids:
            bi, bj = divmod(int(b), kb)
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128].cpu()
            oq, os_ = oracle.quantize_weights_blockwise(blk)
            assert (np_u8(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]) == oq).all()
            assert np_f32_bits(s[bi, bj]) == os_.view(np.uint32)[0, 0]
        # every block's max lands on +-448 (0x7E / 0xFE): a property of all blocks
        blocks = q.view(nb, 128, kb, 128).permute(0, 2, 1, 3).reshape(nb * kb, -1)
        assert bool(((blocks & 0x7F) == 0x7E).any(dim=1).all())
    del ws, qs, ss
    torch.cuda.empty_cache()


@pytest.mark.parametrize("seqs,tokens,heads,hd", [(2, 37, 8, 128), (1, 1, 8, 128), (3, 50, 4, 64),
                                                  (2, 9, 2, 8), (1, 5, 1, 2048), (4, 300, 16, 128),
                                                  (2, 11, 256, 8)])
def test_kv_calibrate_and_given(seqs, tokens, heads, hd):
    dev = device()
    x = workloads.kv_tensor(seed=seqs * tokens, seqs=seqs, tokens=tokens, heads=heads, head_dim=hd)
    xr = x.view(-1, heads, hd)
    qc = Canary(x.numel(), torch.uint8, dev)
    q, s = fp8rl.quantize_kv_fp8(x.to(dev), fp8rl.FP8RL_KV_CALIBRATE, q=qc.view.view(x.shape))
    torch.cuda.synchronize()
    qc.check()
    os_ = oracle.kv_calibrate(xr)
    assert (np_f32_bits(s) == os_.view(np.uint32)).all()
    assert (np_u8(q).reshape(-1, heads, hd) == oracle.kv_quantize(xr, os_)).all()
    # GIVEN with caller scales: ordinary, tiny, huge, zero and negative
    rng = np.random.default_rng(heads)
    cand = np.array([1e-3, 3.7e-2, 1e-30, 1e30, 0.0, -0.5, 2.0 ** -60, 2.0 ** -61, 1e-20, 7.0],
                    dtype=np.float32)
    given = rng.choice(cand, size=heads).astype(np.float32)
    q2, _ = fp8rl.quantize_kv_fp8(x.to(dev), fp8rl.FP8RL_KV_GIVEN,
                                  scales=torch.from_numpy(given).to(dev))
    assert (np_u8(q2).reshape(-1, heads, hd) == oracle.kv_quantize(xr, given)).all()


def test_kv_long_context_full_size():
    """One layer's K for 64 x 20480 tokens x 8 heads x 128: calibrated scales
    bit-exact over the whole tensor, codes on sampled rows."""
    dev = device()
    x = workloads.kv_tensor(seed=5, device=dev)
    q, s = fp8rl.quantize_kv_fp8(x, fp8rl.FP8RL_KV_CALIBRATE)
    torch.cuda.synchronize()
    xr_cpu = x.view(-1, 8, 128).cpu()
    os_ = oracle.kv_calibrate(xr_cpu)
    assert (np_f32_bits(s) == os_.view(np.uint32)).all()
    rows = np.random.default_rng(1).choice(xr_cpu.shape[0], size=4096, replace=False)
    qr = np_u8(q.view(-1, 8, 128)[torch.from_numpy(rows).to(dev)])
    assert (qr == oracle.kv_quantize(xr_cpu[torch.from_numpy(rows)], os_)).all()
    del x, q, xr_cpu
    torch.cuda.empty_cache()


def test_host_streaming_requant_matches_device_path():
    """Host BF16 in, host codes and scales out, through a workspace small enough
    to split tensors across chunks; bit-identical to the device multi-tensor path
    and to the oracle (this is the call the bench's end-to-end figure uses)."""
    dev = device()
    shapes = [(1000, 512), (128, 136), (300, 2048), (7, 8), (640, 1024)]
    ws = [workloads.make_weight(n, k, seed=70 + i) for i, (n, k) in enumerate(shapes)]
    # strided host rows for one tensor (ldw > k, ldq > k)
    big = torch.zeros(300, 2048 + 64, dtype=torch.bfloat16)
    big[:, :2048] = ws[2]
    hw = [w.pin_memory() for w in ws]
    hw[2] = big.pin_memory()[:, :2048]
    qbig = torch.full((300, 2048 + 32), 0x5A, dtype=torch.uint8).pin_memory()
    hq = [torch.empty(w.shape, dtype=torch.uint8).pin_memory() for w in ws]
    hq[2] = qbig[:, :2048]
    hs = [torch.empty((w.shape[0] + 127) // 128, (w.shape[1] + 127) // 128,
                      dtype=torch.float32).pin_memory() for w in ws]
    work = torch.empty(2 * 1_300_000, dtype=torch.uint8, device=dev)       # ~430 rows of k = 1024 per half
    fp8rl.quantize_weights_blockwise_multi_host(hw, hq, hs, work)
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    qd, sd = fp8rl.quantize_weights_blockwise_multi([w.to(dev) for w in ws])
    for i in range(len(ws)):
        assert (hq[i].numpy() == qd[i].cpu().numpy()).all(), i
        assert (hs[i].numpy().view(np.uint32) == sd[i].cpu().numpy().view(np.uint32)).all(), i
        oq, os_ = oracle.quantize_weights_blockwise(ws[i])
        assert (hq[i].numpy() == oq).all(), i
        assert (hs[i].numpy().view(np.uint32) == os_.view(np.uint32)).all(), i
    assert (qbig[:, 2048:].numpy() == 0x5A).all()         # row padding untouched
