"""GPU parity of the truncated importance weights: bit-exact against the
oracle on the pages' workloads, with masks, both clip modes, ragged sizes,
special values, and exhaustively over every binary32 log-ratio."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, device, np_f32_bits

pytestmark = pytest.mark.gpu


def _case(lt, lr, dev, mask=None, c_hi=2.0, c_lo=0.0):
    n = lt.numel()
    wc = Canary(max(n, 1), torch.float32, dev)
    w = wc.view[:n]
    fp8rl.tis_weights(lt.to(dev), lr.to(dev), None if mask is None else mask.to(dev), c_hi, c_lo,
                      w=w)
    torch.cuda.synchronize()
    wc.check()
    ref = oracle.tis_weights(lt.numpy(), lr.numpy(),
                             None if mask is None else mask.numpy(), c_hi, c_lo)
    got = w.cpu().numpy()
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), "first mismatch at %s" % np.argwhere(~same)[:5].ravel()


def test_tiny_workload():
    dev = device()
    lt, lr = workloads.tis_logprobs(4096, seed=0)
    _case(lt, lr, dev)
    _case(lt, lr, dev, c_lo=0.5)
    mask = (torch.arange(4096) % 7 != 3).to(torch.uint8)
    _case(lt, lr, dev, mask=mask)


def test_long_context_student_t_workload():
    dev = device()
    lt, lr = workloads.tis_logprobs(64 * 20480, seed=5, kind="student_t")
    _case(lt, lr, dev)
    _case(lt, lr, dev, c_hi=2.0, c_lo=0.5)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 4097, 1023])
def test_ragged_sizes(n):
    dev = device()
    lt, lr = workloads.tis_logprobs(n, seed=n)
    mask = (torch.arange(n) % 2).to(torch.uint8)
    _case(lt, lr, dev)
    _case(lt, lr, dev, mask=mask)


def test_special_values():
    dev = device()
    v = torch.tensor([0.0, -0.0, float("nan"), float("inf"), -float("inf"), 88.0, 89.0, -87.0,
                      -104.0, -103.9, -150.0, 1e-30, -2.0 ** -25, 0.6931472, 0.69314712],
                     dtype=torch.float32)
    _case(v, torch.zeros_like(v), dev)
    _case(torch.zeros_like(v), v, dev, c_hi=1e30)


def test_every_binary32_log_ratio():
    """lt = every float32 bit pattern, lr = 0, so d = lt exactly; C = 3e38
    (no truncation) so the raw correctly rounded exponential is compared."""
    dev = device()
    chunk = 1 << 28
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=dev).to(torch.int32)
        lt = bits.view(torch.float32)
        w = fp8rl.tis_weights(lt, torch.zeros_like(lt), None, 3e38, 0.0)
        ref = oracle.tis_weights(lt.cpu().numpy(), np.zeros(chunk, np.float32), None, 3e38, 0.0)
        got = w.cpu().numpy()
        same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), "chunk %x: %d mismatches" % (start, (~same).sum())
        del bits, lt, w


# ------------------------------------------------ IS weights + mismatch stats --

def _stats_case(lt, lr, dev, mask=None, c_hi=2.0, c_lo=0.0, mode=fp8rl.FP8RL_IS_TRUNCATE,
                weights=True, loss=None):
    n = lt.numel()
    nst = 5 if loss is None else 6
    wc = Canary(max(n, 1), torch.float32, dev)
    sc = Canary(nst, torch.float64, dev)
    w, st = fp8rl.is_weights_stats(lt.to(dev), lr.to(dev), None if mask is None else mask.to(dev),
                                   c_hi, c_lo, mode, w=wc.view[:n] if weights else None,
                                   stats=sc.view, weights=weights,
                                   loss=None if loss is None else loss.to(dev))
    torch.cuda.synchronize()
    wc.check(); sc.check()
    ref_w, ref_st, terms_abs = oracle.is_weights_stats(lt.numpy(), lr.numpy(),
                                                       None if mask is None else mask.numpy(),
                                                       c_hi, c_lo, mode,
                                                       None if loss is None else loss.numpy())
    if weights:
        got = w.cpu().numpy()
        same = (got.view(np.uint32) == ref_w.view(np.uint32)) | (np.isnan(got) & np.isnan(ref_w))
        assert same.all(), "first mismatch at %s" % np.argwhere(~same)[:5].ravel()
    else:
        assert (wc.view.view(torch.int32).cpu() == wc.view.view(torch.int32).cpu()[0]).all()
    g = st.cpu().numpy()
    # counts exact; sums within the documented bound 2^-20 * sum |terms|
    assert g[0] == ref_st[0] and g[4] == ref_st[4]
    for q in ((1, 2, 3) if loss is None else (1, 2, 3, 5)):
        if not np.isfinite(ref_st[q]):   # inf / NaN terms propagate
            assert g[q] == ref_st[q] or (np.isnan(g[q]) and np.isnan(ref_st[q])), (q, g[q])
            continue
        assert abs(g[q] - ref_st[q]) <= 2.0 ** -20 * terms_abs[q] + 1e-300, (q, g[q], ref_st[q])
    return g, ref_st


@pytest.mark.parametrize("mode", [fp8rl.FP8RL_IS_TRUNCATE, fp8rl.FP8RL_IS_MASK])
def test_is_stats_tiny_and_ragged(mode):
    dev = device()
    for n in (4096, 1, 3, 5, 37, 4099, 70001):
        lt, lr = workloads.tis_logprobs(n, seed=n)
        _stats_case(lt, lr, dev, mode=mode)
        _stats_case(lt, lr, dev, mode=mode, c_lo=0.5)
        mask = (torch.arange(n) % 7 != 3).to(torch.uint8)
        _stats_case(lt, lr, dev, mask=mask, mode=mode)


def test_is_stats_long_context_student_t():
    dev = device()
    lt, lr = workloads.tis_logprobs(64 * 20480, seed=5, kind="student_t")
    for mode in (fp8rl.FP8RL_IS_TRUNCATE, fp8rl.FP8RL_IS_MASK):
        _stats_case(lt, lr, dev, mode=mode)
    _stats_case(lt, lr, dev, mode=fp8rl.FP8RL_IS_MASK, c_lo=0.5, weights=False)


def test_is_stats_special_values_and_empty():
    dev = device()
    lt = torch.tensor([0.0, -1.0, float("nan"), -5.0, 3.0, -100.0, 0.5, -0.5], dtype=torch.float32)
    lr = torch.tensor([0.0, -2.0, -1.0, float("nan"), -90.0, 0.0, 0.5, -0.25], dtype=torch.float32)
    # NaN and huge log-ratios: weights bit-exact, statistics propagate NaN / inf like the oracle
    n = lt.numel()
    w, st = fp8rl.is_weights_stats(lt.to(dev), lr.to(dev), mode=fp8rl.FP8RL_IS_MASK)
    ref_w, ref_st, _ = oracle.is_weights_stats(lt.numpy(), lr.numpy(), mode=oracle.IS_MASK)
    got = w.cpu().numpy()
    assert ((got.view(np.uint32) == ref_w.view(np.uint32)) | (np.isnan(got) & np.isnan(ref_w))).all()
    g = st.cpu().numpy()
    assert g[0] == n and g[4] == ref_st[4]
    assert np.isnan(g[1]) == np.isnan(ref_st[1]) and np.isnan(g[3]) == np.isnan(ref_st[3])
    # valid-only statistics without the NaN tokens
    mask = torch.tensor([1, 1, 0, 0, 1, 1, 1, 1], dtype=torch.uint8)
    _stats_case(lt, lr, dev, mask=mask, mode=fp8rl.FP8RL_IS_MASK)
    # empty input: statistics cleared, nothing written
    e = torch.empty(0, dtype=torch.float32)
    sc = Canary(5, torch.float64, dev)
    fp8rl.is_weights_stats(e.to(dev), e.to(dev), stats=sc.view)
    torch.cuda.synchronize()
    sc.check()
    assert (sc.view.cpu().numpy() == 0).all()


@pytest.mark.parametrize("mode", [fp8rl.FP8RL_IS_TRUNCATE, fp8rl.FP8RL_IS_MASK])
def test_is_stats_weighted_loss(mode):
    """The importance-weighted token loss (sixth statistic) on ragged sizes, with
    and without a mask, and on the long-context Student-t workload."""
    dev = device()
    for n in (1, 5, 4096, 4099, 70001):
        lt, lr = workloads.tis_logprobs(n, seed=100 + n)
        loss = torch.randn(n, generator=torch.Generator().manual_seed(n))
        _stats_case(lt, lr, dev, mode=mode, loss=loss)
        mask = (torch.arange(n) % 3 != 1).to(torch.uint8)
        _stats_case(lt, lr, dev, mask=mask, mode=mode, c_lo=0.5, loss=loss)
    lt, lr = workloads.tis_logprobs(64 * 20480, seed=5, kind="student_t")
    loss = torch.randn(lt.numel(), generator=torch.Generator().manual_seed(9)).abs_()
    g, ref = _stats_case(lt, lr, dev, mode=mode, loss=loss, weights=False)
    assert len(g) == 6
