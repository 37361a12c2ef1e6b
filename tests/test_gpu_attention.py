"""GPU parity of the FP8-KV decode attention against the float64 oracle.

Tolerance, from the arithmetic: the kernel dequantizes exactly (every E4M3
code is an FP16 value) and scales q per head by a power of two before its
FP16 conversion (exact in FP16's normal range), so the score products are
exact and only their FP32 accumulation inside the tensor-core MMA rounds;
exp2 is within 2 ulp; the probabilities, scaled by 2^15 (so FP16 keeps
them normal down to p = 2^-29), are rounded to FP16 (relative 2^-11) for the
weighted sum of V, accumulated in FP32, while the normaliser sums the FP32
probabilities; the result is rounded to BF16.  Per element
|out - o| <= 2^-8 |o| + 1e-3 * sum_t p_t |V_t| (BF16 half-ulp, plus the FP16
probabilities, 2^-11 of the weighted |V|, plus FP32 accumulation), and the
relative Frobenius error against the BF16-rounded oracle is <= 2e-3."""
import math

import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, device

pytestmark = pytest.mark.gpu


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C
    return c


def _check(out, o64, mag, what=""):
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), what
    assert (np.abs(got - o64) <= 2.0 ** -8 * np.abs(o64) + 1e-3 * mag + 1e-30).all(), what
    ref16 = torch.from_numpy(o64).to(torch.bfloat16).double().numpy()
    den = np.linalg.norm(ref16)
    if den > 0:
        assert np.linalg.norm(got - ref16) <= 2e-3 * den, what


def _case(S, Hq, Hkv, T, lens, dev, seed=0, paged=False, page=16):
    rng = np.random.default_rng(seed)
    kc, vc = _codes(rng, (S, T, Hkv, 128)), _codes(rng, (S, T, Hkv, 128))
    ks = rng.uniform(0.002, 0.05, Hkv).astype(np.float32)
    vs = rng.uniform(0.01, 0.2, Hkv).astype(np.float32)
    q = torch.randn(S, Hq, 128, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    o64, mag = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, lens)
    kst, vst = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
    lt = torch.tensor(lens, dtype=torch.int32, device=dev)
    oc = Canary(S * Hq * 128, torch.bfloat16, dev)
    if not paged:
        out = fp8rl.decode_attention_fp8kv(q.to(dev), torch.from_numpy(kc).to(dev),
                                           torch.from_numpy(vc).to(dev), kst, vst, lt,
                                           out=oc.view.view(S, Hq, 128))
    else:
        npg = T // page
        perm = rng.permutation(S * npg)
        kp = np.zeros((S * npg + 3, page, Hkv, 128), np.uint8)
        vp = np.zeros_like(kp)
        table = np.zeros((S, npg), np.int32)
        for s in range(S):
            for j in range(npg):
                dst = perm[s * npg + j] + 3
                kp[dst], vp[dst] = kc[s, j * page:(j + 1) * page], vc[s, j * page:(j + 1) * page]
                table[s, j] = dst
        out = fp8rl.decode_attention_fp8kv(q.to(dev), torch.from_numpy(kp).to(dev),
                                           torch.from_numpy(vp).to(dev), kst, vst, lt,
                                           block_table=torch.from_numpy(table).to(dev),
                                           out=oc.view.view(S, Hq, 128))
    torch.cuda.synchronize()
    oc.check()
    fp8rl.device_status(0)
    _check(out, o64, mag, "S=%d Hq=%d Hkv=%d T=%d paged=%s" % (S, Hq, Hkv, T, paged))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 8), (8, 4), (32, 4)])
def test_contiguous_gqa_groups(hq, hkv):
    _case(3, hq, hkv, 70, [70, 1, 33], device(), seed=hq + hkv)


def test_paged_ragged_and_empty():
    _case(4, 16, 4, 96, [96, 0, 50, 17], device(), seed=5, paged=True, page=16)
    _case(2, 8, 2, 96, [96, 95], device(), seed=6, paged=True, page=32)


@pytest.mark.parametrize("page", [None, 64, 16, 8, 4, 24])
def test_many_stages_every_output(page):
    """64 stages per CTA (4096 tokens) with ragged lengths, contiguous and paged
    (boxes of 64, 16, 8 rows in the swizzled layout; 4 rows plain; page 24 gives
    boxes of 8): every output checked, so that a stage read out of turn shows."""
    dev = device()
    lens = [4096, 4095, 2049, 64, 65, 1]
    if page is None:
        _case(6, 8, 2, 4096, lens, dev, seed=40)
    else:
        T = 4096 + (-4096) % page
        _case(6, 8, 2, T, lens, dev, seed=41 + page, paged=True, page=page)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2)])
def test_many_stages_group_sizes(hq, hkv):
    _case(3, hq, hkv, 3000, [3000, 2999, 1717], device(), seed=50 + hq)


@pytest.mark.parametrize("paged", [False, True])
def test_cluster_split_short_and_long(paged):
    """Few (sequence, head) pairs over long contexts run as clusters of up to 8
    CTAs, each over a range of stages; the short sequence leaves most ranks
    with no stage at all."""
    _case(2, 8, 2, 8192, [8192, 100], device(), seed=60 + int(paged), paged=paged, page=32)


def test_quantized_cache_chain():
    """K and V of 4 sequences x 2048 tokens through the KV quantizer (calibrated
    per-head scales), then decode attention of 32 query heads."""
    dev = device()
    S, T, Hkv, Hq = 4, 2048, 8, 32
    k = workloads.kv_tensor(seed=21, seqs=S, tokens=T, device=dev)
    v = workloads.kv_tensor(seed=22, seqs=S, tokens=T, device=dev)
    kq, ks = fp8rl.quantize_kv_fp8(k, fp8rl.FP8RL_KV_CALIBRATE)
    vq, vs = fp8rl.quantize_kv_fp8(v, fp8rl.FP8RL_KV_CALIBRATE)
    q = torch.randn(S, Hq, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    lens = [2048, 1500, 1, 777]
    out = fp8rl.decode_attention_fp8kv(q.to(dev), kq, vq, ks, vs,
                                       torch.tensor(lens, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    o64, mag = oracle.decode_attention_fp8kv(q, kq.cpu().numpy(), vq.cpu().numpy(),
                                             ks.cpu().numpy(), vs.cpu().numpy(), lens)
    _check(out, o64, mag, "quantized chain")


def test_long_context_sampled_sequences():
    """64 sequences x 20480 tokens x 8 KV heads (the long-context KV workload),
    32 query heads; four sequences checked against the oracle."""
    dev = device()
    S, T, Hkv, Hq = 64, 20480, 8, 32
    k = workloads.kv_tensor(seed=31, device=dev)
    kq, ks = fp8rl.quantize_kv_fp8(k, fp8rl.FP8RL_KV_CALIBRATE)
    del k
    v = workloads.kv_tensor(seed=32, device=dev)
    vq, vs = fp8rl.quantize_kv_fp8(v, fp8rl.FP8RL_KV_CALIBRATE)
    del v
    q = torch.randn(S, Hq, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    lens = torch.full((S,), T, dtype=torch.int32)
    lens[5] = 12345
    out = fp8rl.decode_attention_fp8kv(q.to(dev), kq, vq, ks, vs, lens.to(dev))
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    for s in (0, 5, 31, 63):
        o64, mag = oracle.decode_attention_fp8kv(q[s:s + 1], kq[s].cpu().numpy()[None],
                                                 vq[s].cpu().numpy()[None], ks.cpu().numpy(),
                                                 vs.cpu().numpy(), [int(lens[s])])
        _check(out[s:s + 1], o64, mag, "sequence %d" % s)
    del kq, vq
    torch.cuda.empty_cache()


def test_bad_page_index_is_reported():
    dev = device()
    rng = np.random.default_rng(9)
    kc = torch.from_numpy(_codes(rng, (4, 16, 2, 128))).to(dev)
    vc = torch.from_numpy(_codes(rng, (4, 16, 2, 128))).to(dev)
    sc = torch.full((2,), 0.01, device=dev)
    q = torch.randn(1, 4, 128, device=dev).to(torch.bfloat16)
    table = torch.tensor([[1, 7]], dtype=torch.int32, device=dev)          # page 7 does not exist
    fp8rl.decode_attention_fp8kv(q, kc, vc, sc, sc, torch.tensor([32], dtype=torch.int32,
                                                                device=dev), block_table=table)
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.device_status(0)
    fp8rl.device_status(0)
