"""Pins of the oracle's blockwise-scaled W8A8 GEMM.

* brute force over a 4x4 output tile with exact rational arithmetic
  (fractions.Fraction) at K = 128 and 256: catches a dropped scale, a wrong
  k-block index, or a transposed operand;
* an exactly representable special case (integer-valued codes, power-of-two
  scales): the float64 result must be exact;
* torch.matmul in float64 on the dequantized operands (a library routine);
* the grouped variant equals the dense one on each expert segment, and
  empty segments produce nothing.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_rollout_gb300 import workloads


def _rand_operands(m, n, k, seed):
    rng = np.random.default_rng(seed)
    qa = rng.integers(0, 256, size=(m, k)).astype(np.uint8)
    qw = rng.integers(0, 256, size=(n, k)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x40        # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x41
    sa = rng.uniform(1e-3, 1.0, size=(k // 128, m)).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-2, size=((n + 127) // 128, k // 128)).astype(np.float32)
    return qa, sa, qw, sw


def _exact_value(code):
    c = int(code)
    e, m = (c >> 3) & 0xF, c & 7
    mag = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -mag if c & 0x80 else mag


@pytest.mark.parametrize("k", [128, 256])
def test_brute_force_4x4_exact_rationals(k):
    m, n = 4, 4
    qa, sa, qw, sw = _rand_operands(m, n, k, seed=k)
    y, ab = oracle.gemm_w8a8(qa, sa, qw, sw)
    for i in range(m):
        for j in range(n):
            exact = Fraction(0)
            exact_abs = Fraction(0)
            for kk in range(k):
                a = _exact_value(qa[i, kk]) * Fraction(float(sa[kk // 128, i]))
                w = _exact_value(qw[j, kk]) * Fraction(float(sw[j // 128, kk // 128]))
                exact += a * w
                exact_abs += abs(a) * abs(w)
            # float64 sum of k exact products: error <= k * 2^-53 * sum|terms|
            assert abs(Fraction(float(y[i, j])) - exact) <= Fraction(k, 2 ** 53) * exact_abs
            assert abs(Fraction(float(ab[i, j])) - exact_abs) <= Fraction(k, 2 ** 53) * exact_abs


def test_brute_force_detects_transpose():
    """The 4x4 brute force must distinguish Y from Y^T-style index swaps."""
    qa, sa, qw, sw = _rand_operands(4, 4, 128, seed=11)
    y, _ = oracle.gemm_w8a8(qa, sa, qw, sw)
    assert not np.allclose(y, y.T)


def test_exact_special_case_integer_codes_power_of_two_scales():
    """Codes whose values are small integers and scales that are powers of
    two: every product and partial sum is exact in float64 (and binary32)."""
    rng = np.random.default_rng(12)
    m, n, k = 8, 256, 256
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    ints = np.array([c for c in range(0x7F) if float(table[c]).is_integer() and table[c] <= 8],
                    dtype=np.uint8)
    qa = rng.choice(ints, size=(m, k)) | (rng.integers(0, 2, (m, k)) << 7).astype(np.uint8)
    qw = rng.choice(ints, size=(n, k)) | (rng.integers(0, 2, (n, k)) << 7).astype(np.uint8)
    sa = np.exp2(rng.integers(-3, 2, size=(k // 128, m))).astype(np.float32)
    sw = np.exp2(rng.integers(-3, 2, size=(n // 128, k // 128))).astype(np.float32)
    y, _ = oracle.gemm_w8a8(qa.astype(np.uint8), sa, qw.astype(np.uint8), sw)
    A = oracle.e4m3_decode(qa) * np.repeat(sa.T, 128, axis=1)
    W = oracle.e4m3_decode(qw) * np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1)
    exact = np.array([[sum(Fraction(float(A[i, t])) * Fraction(float(W[j, t])) for t in range(k))
                       for j in range(0, n, 37)] for i in range(m)])
    assert (y[:, ::37] == exact.astype(np.float64)).all()


def test_matches_torch_float64_matmul_on_dequantized_operands():
    a, w = workloads.tiny_linear(seed=0)
    qa, sa = oracle.quantize_act_groupwise(a)
    qw, sw = oracle.quantize_weights_blockwise(w)
    y, ab = oracle.gemm_w8a8(qa, sa, qw, sw)
    A = oracle.e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    W = oracle.e4m3_decode(qw) * np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1)
    ref = (torch.from_numpy(A) @ torch.from_numpy(W).T).numpy()
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * ab.max())
    refab = (torch.from_numpy(np.abs(A)) @ torch.from_numpy(np.abs(W)).T).numpy()
    assert np.allclose(ab, refab, rtol=1e-12)
    # and the quantized product approximates the bf16 product (sanity of the scheme)
    dense = (a.double() @ w.double().T).numpy()
    rel = np.linalg.norm(y - dense) / np.linalg.norm(dense)
    assert rel < 0.1


def test_sampled_rows_cols_equal_full():
    qa, sa, qw, sw = _rand_operands(40, 300, 384, seed=13)
    y, ab = oracle.gemm_w8a8(qa, sa, qw, sw)
    rows, cols = [3, 39, 0, 17], [299, 5, 128, 256, 0]
    ys, abs_ = oracle.gemm_w8a8(qa, sa, qw, sw, rows=rows, cols=cols)
    assert (ys == y[np.ix_(rows, cols)]).all() and (abs_ == ab[np.ix_(rows, cols)]).all()


def test_grouped_equals_dense_per_segment_and_empty_segments():
    rng = np.random.default_rng(14)
    E, n, k = 5, 256, 256
    counts = np.array([3, 0, 130, 0, 7])
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    M = int(off[-1])
    qa, sa, _, _ = _rand_operands(M, n, k, seed=15)
    qw = rng.integers(0, 0x7F, size=(E, n, k)).astype(np.uint8)
    sw = rng.uniform(1e-3, 1e-2, size=(E, n // 128, k // 128)).astype(np.float32)
    y, _ = oracle.grouped_gemm_w8a8(qa, sa, qw, sw, off)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        rows = list(range(r0, r1))
        yd, _ = oracle.gemm_w8a8(qa, sa, qw[e], sw[e], rows=rows)
        assert (y[r0:r1] == yd).all()
    # rows beyond the last segment have no output
    off2 = off.copy()
    off2[-1] = M - 2
    y2, _ = oracle.grouped_gemm_w8a8(qa, sa, qw, sw, off2)
    assert np.isnan(y2[M - 2:]).all() and not np.isnan(y2[:M - 2]).any()


def test_bf16_round_is_rne():
    y = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8 + 2 ** -20)], dtype=np.float64)
    r = oracle.bf16_round(y)
    assert r[0] == 1.0 and r[1] == 1.0 + 2 ** -6 and r[2] == -(1.0 + 2 ** -7)
