"""Pins of the oracle's MoE glue (permute + quantize, SiLU(gate) * up +
quantize), against things other than itself.

The definition is y = BF16_RNE(silu(g) * u): the real product rounded once to
the nearest BF16.  Pins:

* binary32 -> BF16 rounding against torch's cast (a library routine);
* every finite BF16 gate, with several up values: y is the BF16 value nearest
  to the float64 product (checked against its neighbours, wherever float64
  decides it);
* closed forms where float64 cannot decide: for tiny g, silu(g) = g/2 + g^2/4
  + O(g^4) lies strictly above g/2, so a product (g/2) u on a midpoint rounds
  upwards; for large g > 0, silu(g) = g - g e^-g / (1 + e^-g) lies strictly
  below g, so a product g u on a midpoint rounds towards zero;
* signed zeros, infinities and NaN as the IEEE evaluation of g sigma(g) u;
  g <= -256 gives a signed zero; negating u negates y;
* the gather as plain indexing of the token matrix.
"""
import numpy as np
import torch

import oracle
from fp8_precision_rollout_gb300 import workloads


def _f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64_inf_as_2_128(bits):
    """BF16 values with +-inf standing for +-2^128, where round-to-nearest
    overflows (its midpoint with the largest finite value is the threshold)."""
    v = _f64(bits)
    return np.where(np.isinf(v), np.sign(v) * 2.0 ** 128, v)


def _nearest_ok(y_bits, x64):
    """y is at least as close to x as both neighbours in magnitude (x finite)."""
    y = _f64_inf_as_2_128(y_bits)
    s = np.asarray(y_bits, dtype=np.uint32) & 0x8000
    mag = np.asarray(y_bits, dtype=np.uint32) & 0x7FFF
    up = _f64_inf_as_2_128(np.where(mag < 0x7F80, s | (mag + 1), s | mag))
    dn = _f64_inf_as_2_128(np.where(mag > 0, s | (mag - 1), s | mag))
    d = np.abs(y - x64)
    return (d <= np.abs(up - x64)) & (d <= np.abs(dn - x64))


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


def _silu64(g):
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        pos = g / (1.0 + np.exp(-g))
        e = np.exp(np.minimum(g, 0.0))
        neg = g * e / (1.0 + e)
    return np.where(g > 0, pos, neg)


def test_silu_mul_nearest_over_every_finite_gate():
    """All finite BF16 gates x several up values: y is the BF16 value nearest
    the float64 product wherever that product is not within 2^-30 of a
    midpoint (float64 decides those; the rest are pinned by closed forms)."""
    gb = np.arange(1 << 16, dtype=np.uint32)
    gf = _f64(gb)
    fin = np.isfinite(gf) & (gf != 0)
    gb, gf = gb[fin], gf[fin]
    for ub in (0x3F80, 0x3FC0, 0xBFA3, 0x4131, 0x3E55, 0x5F01, 0x2001):
        y = oracle.silu_mul_pairs(gb.astype(np.uint16), np.full(gb.size, ub, np.uint16))
        x = _silu64(gf) * _f64(ub)
        ok = _nearest_ok(y, x)
        # product within 2^-30 (relative) of a BF16 midpoint: float64 cannot decide
        mag = np.abs(x)
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
        q = 2.0 ** (np.maximum(e, -126) - 7)
        t = mag / q
        near = np.abs(t - np.floor(t) - 0.5) <= t * 2.0 ** -30
        small = mag < 2.0 ** -134 * (1 - 2.0 ** -20)      # rounds to a signed zero
        assert (ok | near).all(), (ub, gf[~(ok | near)][:5])
        assert ((y[small] & 0x7FFF) == 0).all()
        assert near.mean() < 0.25     # structural midpoints: large and tiny gates (closed forms)


def test_silu_mul_tiny_gate_closed_form():
    """|g| < 2^-60: silu(g) = g/2 + g^2/4 - ..., strictly above g/2.  With u = 1
    a subnormal g of odd mantissa puts g/2 on a midpoint: y is the BF16 value
    above it (larger for g > 0, smaller in magnitude for g < 0); otherwise
    y = g/2."""
    for sign in (0, 0x8000):
        gb = (sign | np.arange(1, 67 << 7, dtype=np.uint32)).astype(np.uint16)
        g = _f64(gb)
        assert (np.abs(g) < 2.0 ** -60).all()
        y = oracle.silu_mul_pairs(gb, np.full(gb.size, 0x3F80, np.uint16)).astype(np.uint32)
        half = g / 2                                   # exact in binary32
        hb = half.astype(np.float32).view(np.uint32) >> 16   # |g/2| truncated to BF16
        exact = _f64(hb) == half
        assert (~exact).sum() > 0
        assert (y[exact] == hb[exact]).all()
        want = hb[~exact] + 1 if sign == 0 else hb[~exact]  # the neighbour towards +inf
        assert (y[~exact] == want).all()


def test_silu_mul_large_gate_closed_form():
    """g >= 64: silu(g) lies strictly between g (1 - 2^-90) and g.  With u = 1.5
    and g of even mantissa (at most 7 significant bits), every product g u is a
    BF16 value or a midpoint; a midpoint rounds towards zero, a representable
    product is returned as it is."""
    gb = np.arange(0x4280, 0x7F80, 2, dtype=np.uint32)          # [64, max finite], even mantissa
    g = _f64(gb)
    y = oracle.silu_mul_pairs(gb.astype(np.uint16), np.full(gb.size, 0x3FC0, np.uint16))
    x = g * 1.5                                                   # exact in float64
    xf = x.astype(np.float32)
    fin = np.isfinite(xf)
    xb = xf[fin].view(np.uint32)
    rep = (xb & 0xFFFF) == 0
    mid = (xb & 0xFFFF) == 0x8000
    assert (rep | mid).all()
    yy = y[fin]
    assert (yy[rep] == (xb[rep] >> 16)).all()
    assert (yy[mid] == (xb[mid] >> 16)).all()                    # truncation: towards zero
    assert (y[~fin] == 0x7F80).all()                              # beyond BF16 max: +inf


def test_silu_mul_structural_midpoints_match_decimal():
    """The oracle settles exact float64 midpoints of large and tiny gates by the
    sign of silu's remainder; an 80-digit decimal evaluation agrees on a sample."""
    rng = np.random.default_rng(44)
    big = rng.integers(0x4240, 0x7F80, size=300)                 # g in [48, max]
    tiny = rng.integers(1, 0x1B00, size=300) | rng.integers(0, 2, size=300) * 0x8000
    for gb in np.concatenate([big, tiny]).astype(np.uint16):
        for ub in (0x3FC0, 0xBFA0, 0x4330, 0x3F81):
            y = int(oracle.silu_mul_pairs(np.array([gb]), np.array([ub], np.uint16))[0])
            d = oracle.silu_mul_decimal(int(gb), ub, y)
            assert y == d, (hex(gb), hex(ub), hex(y), hex(d))


def test_silu_mul_special_values():
    P0, N0, PI, NI, NAN = 0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0
    one, m_one, big_neg = 0x3F80, 0xBF80, 0xC400                  # 1, -1, -512
    cases = [(P0, one, P0), (N0, one, N0), (P0, m_one, N0), (N0, m_one, P0),
             (P0, PI, NAN), (PI, one, PI), (PI, m_one, NI), (PI, P0, NAN), (NI, one, NAN),
             (one, PI, PI), (one, NI, NI), (one, P0, P0), (one, N0, N0), (m_one, P0, N0),
             (big_neg, one, N0), (big_neg, m_one, P0), (big_neg, PI, NI), (0x7FC1, one, NAN),
             (one, 0xFFC0, NAN)]
    g = np.array([c[0] for c in cases], dtype=np.uint16)
    u = np.array([c[1] for c in cases], dtype=np.uint16)
    y = oracle.silu_mul_pairs(g, u)
    for (gi, ui, want), got in zip(cases, y):
        if want == NAN:
            assert (got & 0x7F80) == 0x7F80 and (got & 0x7F), (hex(gi), hex(ui), hex(got))
        else:
            assert got == want, (hex(gi), hex(ui), hex(got), hex(want))
    # every g <= -256 gives a signed zero for every finite u
    gb = np.arange(0xC380, 0xFF80, dtype=np.uint32).astype(np.uint16)
    for ub in (0x3F80, 0x7F7F, 0xFF7F):
        yy = oracle.silu_mul_pairs(gb, np.full(gb.size, ub, np.uint16))
        assert ((yy & 0x7FFF) == 0).all() and (((yy & 0x8000) != 0) == (ub < 0x8000)).all()


def test_silu_mul_sign_symmetry_in_up():
    rng = np.random.default_rng(41)
    g = rng.integers(0, 1 << 16, size=200_000).astype(np.uint16)
    u = rng.integers(0, 1 << 15, size=200_000).astype(np.uint16)
    y1 = oracle.silu_mul_pairs(g, u)
    y2 = oracle.silu_mul_pairs(g, u | 0x8000)
    nan = ((y1 & 0x7F80) == 0x7F80) & ((y1 & 0x7F) != 0)
    assert (y2[~nan] == (y1[~nan] ^ 0x8000)).all()


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
