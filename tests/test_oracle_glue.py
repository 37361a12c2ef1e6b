"""Pins of the oracle's MoE glue (permute + quantize, SiLU(gate) * up +
quantize), against things other than itself:

* the glue exponential against float64 exp on a dense sweep of binary32
  inputs (at most 2 ulp), with its stated domain ends;
* binary32 -> BF16 rounding against torch's cast (a library routine);
* silu(g) * u over every finite BF16 gate value against the float64 SiLU
  (at most one BF16 ulp apart, equal almost everywhere);
* the gather as plain indexing of the token matrix.
"""
import numpy as np
import torch

import oracle
from fp8_precision_rollout_gb300 import workloads


def _ulps(got32, ref64):
    ref32 = ref64.astype(np.float32)
    up = np.abs(np.nextafter(ref32, np.float32(np.inf)) - ref32).astype(np.float64)
    return np.abs(got32.astype(np.float64) - ref64) / up


def test_glue_exp_accuracy_dense_sweep():
    lo = np.float32(-86.0).view(np.uint32)
    # every 37th binary32 in [-86, 0) and in [0, 88]: ~60 M inputs
    neg = np.arange(np.uint32(0x80000000), lo, 37, dtype=np.uint32).view(np.float32)
    pos = np.arange(0, np.float32(88.0).view(np.uint32), 37, dtype=np.uint32).view(np.float32)
    for x in (neg, pos):
        e = oracle.glue_exp32(x)
        u = _ulps(e, np.exp(x.astype(np.float64)))
        assert u.max() <= 2.0, (u.max(), x[np.argmax(u)])


def test_glue_exp_special_values_and_domain():
    x = np.array([0.0, -0.0, 1.0, np.nan, 88.0001, 1e30, -86.0001, -1e30], dtype=np.float32)
    e = oracle.glue_exp32(x)
    assert e[0] == 1.0 and e[1] == 1.0
    assert abs(float(e[2]) - np.e) <= 2.0 ** -22 * np.e
    assert np.isnan(e[3]) and np.isinf(e[4]) and np.isinf(e[5]) and e[6] == 0.0 and e[7] == 0.0
    # below -86 the true value is < 2^-124, so 1 + e^x rounds to 1 either way
    assert np.float32(1.0) + np.float32(np.exp(-86.0)) == np.float32(1.0)


def test_float_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(40)
    bits = rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000            # exact ties
    bits[1000:2000] = (bits[1000:2000] & 0xFFFF0000) | 0x7FFF
    x = bits.view(np.float32)
    ours = oracle.float_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert (ours[~nan] == ref[~nan]).all()
    assert ((ours[nan] & 0x7F80) == 0x7F80).all() and ((ours[nan] & 0x7F) != 0).all()


def test_silu_over_every_bf16_gate():
    g_bits = np.arange(1 << 16, dtype=np.uint16)
    g = g_bits.view(np.int16)
    gt = torch.from_numpy(g.copy()).view(torch.bfloat16)
    finite = torch.isfinite(gt.float()).numpy()
    gt, gf = gt[torch.from_numpy(finite)], gt.float().numpy()[finite].astype(np.float64)
    h = torch.cat([gt.view(1, -1), torch.ones_like(gt).view(1, -1)], dim=1)    # up = 1
    y = oracle.silu_mul_bf16(h).float().numpy().reshape(-1).astype(np.float64)
    with np.errstate(over="ignore"):
        silu64 = gf / (1.0 + np.exp(-gf))
    ref = torch.from_numpy(silu64).to(torch.bfloat16).double().numpy()
    deep = gf < -88.0                      # the stated domain end: e^-g -> inf, silu -> -0
    assert (y[deep] == 0).all()
    ok = ~deep
    diff = np.abs(y[ok] - ref[ok])
    assert (diff <= 2.0 ** -7 * np.abs(ref[ok]) + 1e-40).all()   # one BF16 ulp at most
    assert (diff == 0).mean() > 0.999


def test_silu_mul_is_elementwise_and_uses_up():
    h = workloads.expert_inputs(7, 512, seed=3)                  # [gate 256 | up 256]
    y = oracle.silu_mul_bf16(h)
    perm = np.random.default_rng(1).permutation(256)
    hp = torch.cat([h[:, :256][:, perm], h[:, 256:][:, perm]], dim=1)
    assert (oracle.silu_mul_bf16(hp).view(torch.int16) == y[:, perm].view(torch.int16)).all()
    h2 = h.clone()
    h2[:, 256:] = -h2[:, 256:]                                    # negating up negates y
    y2 = oracle.silu_mul_bf16(h2)
    assert (y2.float() == -y.float()).all()


def test_gather_is_indexing():
    a = workloads.dense_acts(50, 640, seed=4)
    rows = np.array([49, 0, 0, 17, 3, 49, 25])
    q, s = oracle.quantize_act_gather(a, rows)
    for i, r in enumerate(rows):
        qr, sr = oracle.quantize_act_groupwise(a[r:r + 1])
        assert (q[i] == qr[0]).all() and (s[:, i] == sr[:, 0]).all()
