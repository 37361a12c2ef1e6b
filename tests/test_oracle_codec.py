"""Pins of the oracle's E4M3 codec against things other than itself.

* the format facts the FP8-RL pages print (golden/e4m3_format.json),
* torch's float8_e4m3fn decode (a library special case),
* counting properties of the encoding (OCP E4M3: 126 positive finite
  non-zero codes, max 448 = 0x7E, min subnormal 2^-9 = 0x01),
* exhaustive nearest-value brute force over the decoded table on every
  binary32 in the range where rounding is non-trivial,
* torch's binary32 -> float8_e4m3fn cast on pre-clamped values.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle


def test_format_facts_from_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_format.json")))
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = vals[np.isfinite(vals)]
    assert finite.max() == g["max_finite"]
    pos = finite[finite > 0]
    assert pos[pos >= g["min_normal"]].min() == g["min_normal"]
    # smallest normal is the start of the exponent range: 2^(1-bias) with bias 2^(e-1)-1
    bias = 2 ** (g["exponent_bits"] - 1) - 1
    assert g["min_normal"] == 2.0 ** (1 - bias)
    # "about 1 part in 8": the spacing at the start of each binade, relative
    normals = np.unique(pos[pos >= g["min_normal"]])
    rel = np.diff(normals) / normals[:-1]
    assert rel.max() == g["relative_step_at_binade_start"]
    assert 2 ** g["mantissa_bits"] == 8


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_decode(codes.numpy())
    nan_ref, nan_ours = np.isnan(ref), np.isnan(ours)
    assert (nan_ref == nan_ours).all()
    assert set(np.nonzero(nan_ours)[0]) == {0x7F, 0xFF}
    fin = ~nan_ref
    assert (ref[fin] == ours[fin]).all()
    assert (np.signbit(ref[fin]) == np.signbit(ours[fin])).all()


def test_code_counts():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    pos = [c for c in range(256) if np.isfinite(vals[c]) and vals[c] > 0]
    assert len(pos) == 126
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert vals[0x80] == 0.0 and np.signbit(vals[0x80])
    # monotone within each sign
    assert (np.diff(vals[0x00:0x7F]) > 0).all()
    assert (np.diff(vals[0x80:0xFF]) < 0).all()


def test_encode_decode_identity():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert (oracle.e4m3_encode(vals) == codes).all()


def test_midpoints_tie_to_even():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        mid = np.float32((vals[c] + vals[c + 1]) / 2)     # exact: <= 5 significant bits
        assert float(mid) == (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == want
        assert oracle.e4m3_encode(np.array([-mid]))[0] == (0x80 | want)


def test_saturation_and_signed_zero():
    big = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e30, np.inf], dtype=np.float32)
    assert (oracle.e4m3_encode(big) == 0x7E).all()
    assert (oracle.e4m3_encode(-big) == 0xFE).all()
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    tiny = np.array([0.0, 1e-30, 2.0 ** -11, 2.0 ** -10], dtype=np.float32)
    assert (oracle.e4m3_encode(tiny) == 0x00).all()
    assert (oracle.e4m3_encode(-tiny) == 0x80).all()
    above = np.nextafter(np.float32(2.0 ** -10), np.float32(1))
    assert oracle.e4m3_encode(np.array([above]))[0] == 0x01


def _brute_force(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value by table search, ties to the even code, saturating."""
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))       # 0 .. 448 ascending
    a = np.abs(x.astype(np.float64))
    i = np.clip(np.searchsorted(table, a), 1, 0x7E)
    lo, hi = table[i - 1], table[i]
    dlo, dhi = a - lo, hi - a
    code = np.where(dlo < dhi, i - 1, np.where(dhi < dlo, i, np.where((i - 1) % 2 == 0, i - 1, i)))
    code = np.where(a >= 448.0, 0x7E, code)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def test_encode_exhaustive_vs_brute_force():
    # every positive binary32 in [2^-12, 2^10): all rounding decisions live here
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(2.0 ** 10).view(np.uint32)
    step = 1 << 24
    for start in range(int(lo), int(hi), step):
        bits = np.arange(start, min(start + step, int(hi)), dtype=np.uint32)
        x = bits.view(np.float32)
        assert (oracle.e4m3_encode(x) == _brute_force(x)).all()
    # and a sample of everything else, both signs
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    assert (oracle.e4m3_encode(x) == _brute_force(x)).all()


def test_encode_matches_torch_cast_on_clamped_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(3_000_000) * np.exp2(rng.uniform(-14, 10, 3_000_000))).astype(np.float32)
    xc = np.clip(x, -448.0, 448.0)
    ref = torch.from_numpy(xc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (oracle.e4m3_encode(x) == ref).all()


@pytest.mark.parametrize("j", [-20, -9, -1, 0, 3, 17])
def test_exact_round_trip_of_representable_blocks(j):
    """A group of E4M3 values times 2^j whose max is 448*2^j has scale 2^j,
    codes equal to the original codes, and dequantizes bit-exactly."""
    rng = np.random.default_rng(j + 100)
    codes = rng.integers(0, 0x7F, size=128).astype(np.uint8)
    codes[rng.integers(0, 128)] = 0x7E
    codes |= (rng.integers(0, 2, size=128) << 7).astype(np.uint8)
    vals = oracle.e4m3_decode(codes) * 2.0 ** j
    a = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    assert (a.to(torch.float64).numpy() == vals).all()           # representable in bf16
    q, s = oracle.quantize_act_groupwise(a.view(1, 128))
    assert s[0, 0] == np.float32(2.0 ** j)
    # -0 codes come back as 0x80 and +0 as 0x00
    assert (q[0] == codes).all()
    assert (oracle.e4m3_decode(q[0]) * np.float64(s[0, 0]) == vals).all()
