"""Pins of the oracle's truncated importance weights.

* closed forms the pages' definition fixes (golden/tis_closed_forms.json);
* correct rounding: the C float64 path plus decimal resolution agrees with a
  pure-Python 60-digit decimal exponential on samples spanning the domain,
  including every input the float64 path flagged as near a rounding boundary;
* the weight is the ratio of probabilities: for probabilities given exactly
  as binary32 numbers, w agrees with p_train / p_rollout to the accuracy the
  logs allow;
* clip semantics: NaN propagates, the mask zeroes, C and 1/C bound the result.
"""
import json
import math
import os

import numpy as np

import oracle
from fp8_precision_rollout_gb300 import workloads


def test_closed_forms(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tis_closed_forms.json")))
    for c in g["cases"]:
        lt = np.array([c["logp_train"]], dtype=np.float32)
        lr = np.array([c["logp_rollout"]], dtype=np.float32)
        w = oracle.tis_weights(lt, lr, c_hi=g["C"], c_lo=c["c_lo"])[0]
        if "w_hex" in c:
            assert hex(int(np.float32(w).view(np.uint32))) == hex(int(c["w_hex"], 16)), c["why"]
        else:
            assert w == np.float32(c["w"]), c["why"]


def test_correct_rounding_against_decimal():
    rng = np.random.default_rng(20)
    parts = [
        rng.uniform(-104, 0.7, 3000),
        rng.normal(0, 0.05, 3000),
        rng.normal(0, 1e-6, 1000),
        np.ldexp(rng.uniform(0.5, 1, 1000), rng.integers(-40, -20, 1000)) * rng.choice([-1, 1], 1000),
        rng.uniform(85, 90, 500),
        rng.uniform(-104.5, -87, 500),
    ]
    d = np.concatenate(parts).astype(np.float32)
    e = oracle.tis_exp(d, np.zeros_like(d))
    for di, ei in zip(d, e):
        assert np.float32(ei).view(np.uint32) == oracle.exp_rn32_decimal(di).view(np.uint32), di


def test_flagged_boundary_cases_are_resolved_exactly():
    # near 0, e^d sits close to binary32 midpoints (e.g. d = -2^-25 is 2^-51 above one)
    d = np.array([-2.0 ** -25, 2.0 ** -24, -3 * 2.0 ** -25, 2.0 ** -30], dtype=np.float32)
    e = oracle.tis_exp(d, np.zeros_like(d))
    assert oracle.tis_exp.last_hard_count >= 1
    for di, ei in zip(d, e):
        assert ei == oracle.exp_rn32_decimal(di)
    assert e[0] == np.float32(1.0)               # 1 - 2^-25 + 2^-51 is above the midpoint
    # dense sweep: all floats in a window around 0 where many inputs are flagged
    bits = np.arange(np.float32(2.0 ** -26).view(np.uint32), np.float32(2.0 ** -26).view(np.uint32) + 20000,
                     dtype=np.uint32)
    d = np.concatenate([bits.view(np.float32), -bits.view(np.float32)])
    e = oracle.tis_exp(d, np.zeros_like(d))
    sample = np.random.default_rng(21).choice(d.size, 400, replace=False)
    for i in sample:
        assert e[i] == oracle.exp_rn32_decimal(d[i])


def test_weight_is_probability_ratio():
    rng = np.random.default_rng(22)
    p_roll = rng.uniform(1e-4, 1, 2000)
    p_train = np.clip(p_roll * np.exp(rng.normal(0, 0.3, 2000)), 1e-6, 1)
    lt = np.log(p_train).astype(np.float32)
    lr = np.log(p_roll).astype(np.float32)
    w = oracle.tis_weights(lt, lr, c_hi=1e30)
    ratio = p_train / p_roll
    # log-probs carry binary32 rounding (|log p| <= ~14): allow that in the exponent
    tol = (np.abs(np.log(p_train)) + np.abs(np.log(p_roll))) * 2.0 ** -23 + 2.0 ** -22
    assert (np.abs(w / ratio - 1) <= tol * 1.01).all()


def test_clip_mask_nan():
    lt, lr = workloads.tis_logprobs(4096, seed=0)
    lt, lr = lt.numpy(), lr.numpy()
    e = oracle.tis_exp(lt, lr)
    w1 = oracle.tis_weights(lt, lr)
    assert (w1 <= 2).all() and (w1 == np.minimum(e, np.float32(2))).all()
    w2 = oracle.tis_weights(lt, lr, c_lo=0.5)
    assert (w2 >= 0.5).all() and (w2 <= 2).all()
    mask = (np.arange(4096) % 3 != 0).astype(np.uint8)
    w3 = oracle.tis_weights(lt, lr, mask=mask)
    assert (w3[mask == 0] == 0).all() and (w3[mask == 1] == w1[mask == 1]).all()
    nan = np.array([np.nan, 0.0], dtype=np.float32)
    w4 = oracle.tis_weights(nan, np.zeros(2, np.float32))
    assert math.isnan(w4[0]) and w4[1] == 1.0
    inf = np.array([np.inf, -np.inf], dtype=np.float32)
    w5 = oracle.tis_weights(inf, np.zeros(2, np.float32))
    assert w5[0] == 2.0 and w5[1] == 0.0


# ------------------------------------------------ IS weights + mismatch stats --

def test_is_stats_closed_forms():
    """lt == lr: every ratio is 1, both KL estimates 0, nothing clipped."""
    lt = np.linspace(-20, -0.01, 1000).astype(np.float32)
    for mode in (oracle.IS_TRUNCATE, oracle.IS_MASK):
        w, st, _ = oracle.is_weights_stats(lt, lt.copy(), mode=mode)
        assert (w == 1).all()
        assert list(st) == [1000.0, 0.0, 0.0, 1000.0, 0.0]


def test_is_stats_constant_shift_matches_exponential():
    """d = c for every token: k1 = -c n, sum e = n RN32(e^c), k3 = n fl32(fl32(e - 1) - c);
    with c = 1 (e > 2) TIS clips every token to 2 and MIS masks every token."""
    n, c = 777, np.float32(1.0)
    lr = np.full(n, -3.0, np.float32)
    lt = (lr + c).astype(np.float32)
    e1 = np.float32(np.exp(np.float64(1.0)))                # correctly rounded here (checked below)
    assert e1 == oracle.exp_rn32_decimal(np.float32(1.0))
    w, st, _ = oracle.is_weights_stats(lt, lr)
    assert (w == 2).all() and st[4] == n
    assert st[1] == -float(c) * n
    assert st[3] == float(e1) * n
    assert st[2] == float(np.float32(np.float32(e1 - np.float32(1)) - c)) * n
    w, st, _ = oracle.is_weights_stats(lt, lr, mode=oracle.IS_MASK)
    assert (w == 0).all() and st[4] == n


def test_is_stats_mask_and_ranges():
    lt, lr = workloads.tis_logprobs(5000, seed=3)
    lt, lr = lt.numpy(), lr.numpy()
    e = oracle.tis_exp(lt, lr)
    mask = (np.arange(5000) % 5 != 0).astype(np.uint8)
    w, st, _ = oracle.is_weights_stats(lt, lr, mask=mask, mode=oracle.IS_MASK, c_lo=0.5)
    keep = (e >= 0.5) & (e <= 2) & (mask == 1)
    assert (w[keep] == e[keep]).all() and (w[~keep] == 0).all()
    assert st[0] == mask.sum() and st[4] == ((~((e >= 0.5) & (e <= 2))) & (mask == 1)).sum()
    # excluded tokens do not contribute: same stats as the oracle on the kept subset
    _, st2, _ = oracle.is_weights_stats(lt[mask == 1], lr[mask == 1], mode=oracle.IS_MASK, c_lo=0.5)
    assert (st == st2).all()
    # TIS weights equal tis_weights (same clip), and k1 = -(sum of d) exactly
    w_t, st_t, _ = oracle.is_weights_stats(lt, lr, mask=mask)
    assert (w_t == oracle.tis_weights(lt, lr, mask=mask)).all()
    d = (lt - lr).astype(np.float32)
    assert st_t[1] == -math.fsum(d[mask == 1].astype(np.float64).tolist())


def test_is_stats_estimate_kl_of_gaussian_shift():
    """Log-ratios d ~ N(0, s^2) with tokens drawn under the rollout policy: the
    k3 mean estimates E[e^d - 1 - d] = exp(s^2/2) - 1, the ratio mean E[e^d] =
    exp(s^2/2), the k1 mean E[-d] = 0 (standard errors from the sample)."""
    rng = np.random.default_rng(31)
    n, s = 400_000, 0.1
    lr = -np.abs(rng.normal(0, 2, n)).astype(np.float32)
    d = rng.normal(0, s, n)
    lt = (lr.astype(np.float64) + d).astype(np.float32)
    _, st, _ = oracle.is_weights_stats(lt, lr, c_hi=1e30)
    dd = (lt - lr).astype(np.float64)
    want_ratio = math.exp(s * s / 2)
    assert abs(st[3] / n - want_ratio) < 5 * np.std(np.exp(dd)) / math.sqrt(n)
    assert abs(st[2] / n - (want_ratio - 1)) < 5 * np.std(np.exp(dd) - 1 - dd) / math.sqrt(n)
    assert abs(st[1] / n) < 5 * s / math.sqrt(n)
    # k3 terms are non-negative wherever |d| is large enough to dominate rounding
    e = oracle.tis_exp(lt, lr)
    k3 = ((e - np.float32(1)).astype(np.float32) - (lt - lr).astype(np.float32)).astype(np.float32)
    big = np.abs((lt - lr).astype(np.float32)) >= 2.0 ** -9
    assert (k3[big] > 0).all()


def test_is_stats_weighted_loss_closed_forms():
    """Sixth statistic, sum of fl32(w * loss) over the valid tokens: lt == lr gives
    w = 1 (the plain loss sum); d >= ln 2 gives w = 2 under TIS and 0 under MIS;
    masked-out tokens never count; one token is the product itself."""
    rng = np.random.default_rng(41)
    n = 999
    lt = rng.uniform(-20, -0.1, n).astype(np.float32)
    loss = rng.normal(0, 1, n).astype(np.float32)
    _, st, ta = oracle.is_weights_stats(lt, lt.copy(), loss=loss)
    assert len(st) == 6 and st[5] == math.fsum(loss.astype(np.float64).tolist())
    assert ta[5] == math.fsum(np.abs(loss).astype(np.float64).tolist())
    lr = (lt - np.float32(1.0)).astype(np.float32)            # d = 1 > ln 2 for every token
    assert ((lt - lr).astype(np.float32) >= np.float32(0.6932)).all()
    _, st, _ = oracle.is_weights_stats(lt, lr, loss=loss)
    assert st[5] == math.fsum((2.0 * loss.astype(np.float64)).tolist())
    _, st, _ = oracle.is_weights_stats(lt, lr, loss=loss, mode=oracle.IS_MASK)
    assert st[5] == 0.0
    mask = (np.arange(n) % 4 == 0).astype(np.uint8)
    _, st, _ = oracle.is_weights_stats(lt, lt.copy(), mask=mask, loss=loss)
    assert st[5] == math.fsum(loss[mask == 1].astype(np.float64).tolist())
    # one token: the rounded product of its weight and loss
    w, st, _ = oracle.is_weights_stats(lt[:1], (lt[:1] + np.float32(0.3)).astype(np.float32),
                                       loss=np.float32([3.0]))
    assert st[5] == float(np.float32(w[0] * np.float32(3.0)))
    # without a loss the statistics keep five entries
    assert len(oracle.is_weights_stats(lt, lt.copy())[1]) == 5
