"""CPU oracle for the FP8 rollout hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct restatement of what the library computes, used
by the tests, by ``__graft_entry__.smoke()`` and by the benchmark's CPU
baseline leg.  The product path (the CUDA library and its Python binding)
never imports this package, and this package never imports the product.

The arithmetic lives in ``fp8rl_oracle.cpp`` (plain C++, one IEEE operation
per step, no fast-math, no FMA contraction); this module marshals numpy arrays
into it and adds the few steps that are clearer in Python:

* the exact resolution of the rare TIS inputs whose binary32 rounding the
  float64 ``exp`` cannot decide (a 60-digit ``decimal`` exponential), and of
  the rare MoE-glue products silu(g) * u that lie too close to a BF16
  rounding midpoint for float64 (80-digit ``decimal``),
* the clip / mask of the TIS weights (numpy ``where``), and
* the BF16 rounding of float64 GEMM outputs (a torch CPU cast).

Each function names the passage of the FP8-RL pages it follows (summary page,
sections 3.4.1-3.4.4; E4M3 per Micikevicius et al.).

Parity status: every function here is pinned by tests/test_oracle_*.py except
two readings the pages leave open, which are parity unpinned: the KV scale
formula (per-head amax/448; section 3.4.4 gives no formula, so only its
arithmetic, not the choice of formula, is pinned) and the Zipf form of the
MoE routing bias in the synthetic inputs (input generation, not method).
"""
from __future__ import annotations

import ctypes
import math
import os
from decimal import Decimal, localcontext

import numpy as np

from . import build as _build

_LIB = None


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [f32]
        L.orc_e4m3_encode_array.argtypes = [P, P, i64, ctypes.c_int]
        L.orc_e4m3_decode_array.argtypes = [P, P, i64]
        L.orc_quantize_values.argtypes = [P, P, P, i64, ctypes.c_int]
        L.orc_quantize_weights_blockwise.argtypes = [P, i64, i64, i64, P, i64, P, ctypes.c_int]
        L.orc_quantize_act_groupwise.argtypes = [P, i64, i64, i64, P, P, ctypes.c_int]
        L.orc_kv_calibrate.argtypes = [P, i64, ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
        L.orc_kv_quantize.argtypes = [P, i64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
        L.orc_gemm_w8a8_sampled.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P, i64, P, P,
                                            ctypes.c_int]
        L.orc_grouped_gemm_w8a8_sampled.argtypes = [P, P, P, P, P, i32, i64, i64, i64, P, i64,
                                                    P, i64, P, P, ctypes.c_int]
        L.orc_tis_exp.restype = i64
        L.orc_tis_exp.argtypes = [P, P, i64, P, P, i64, ctypes.c_int]
        L.orc_float_to_bf16.argtypes = [P, P, i64]
        L.orc_silu_mul_pairs.restype = i64
        L.orc_silu_mul_pairs.argtypes = [P, P, i64, P, P, i64, ctypes.c_int]
        L.orc_silu_mul_bf16.restype = i64
        L.orc_silu_mul_bf16.argtypes = [P, i64, i64, i64, P, P, i64, ctypes.c_int]
        _LIB = L
    return _LIB


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """BF16 data as its uint16 bit patterns (numpy has no bf16)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                        .view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    assert a.dtype == np.uint16, "BF16 inputs are torch.bfloat16 tensors or uint16 bit arrays"
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------ codec --

def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (float64; NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode_array(_p(c), _p(out), c.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code of each binary32 value: RNE, saturating at +-448, sign kept."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(x), _p(out), x.size, threads())
    return out


def quantize_values(x, s) -> np.ndarray:
    """Code of binary32 x under binary32 scale s: E4M3(fl32(x / s)); s == 0 keeps +-0."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    s = np.ascontiguousarray(np.broadcast_to(np.asarray(s, dtype=np.float32), x.shape))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_quantize_values(_p(x), _p(s), _p(out), x.size, threads())
    return out


# ------------------------------------------------------------- quantizers --

def quantize_weights_blockwise(w):
    """128x128-block E4M3 quantization of a BF16 [n, k] matrix.

    Returns (codes uint8 [n, k], scales float32 [ceil(n/128), ceil(k/128)]).
    """
    wb = _u16(w)
    n, k = wb.shape
    q = np.zeros((n, k), dtype=np.uint8)
    s = np.zeros(((n + 127) // 128, (k + 127) // 128), dtype=np.float32)
    lib().orc_quantize_weights_blockwise(_p(wb), n, k, k, _p(q), k, _p(s), threads())
    return q, s


def quantize_act_groupwise(a):
    """Per-token 1x128-group E4M3 quantization of a BF16 [m, k] matrix.

    Returns (codes uint8 [m, k], scales float32 [ceil(k/128), m] group-major).
    """
    ab = _u16(a)
    m, k = ab.shape
    q = np.zeros((m, k), dtype=np.uint8)
    s = np.zeros(((k + 127) // 128, m), dtype=np.float32)
    lib().orc_quantize_act_groupwise(_p(ab), m, k, k, _p(q), _p(s), threads())
    return q, s


def quantize_act_gather(a, rows):
    """MoE glue, permute + quantize: the expert-sorted rows a[rows[r]] of the
    token matrix a, quantized in 1x128 groups (quantize_act_groupwise of the
    gathered matrix)."""
    import torch
    idx = np.asarray(rows, dtype=np.int64)
    ab = _u16(a)
    return quantize_act_groupwise(torch.from_numpy(np.ascontiguousarray(ab[idx])).view(torch.bfloat16))


def float_to_bf16(x) -> np.ndarray:
    """binary32 -> BF16 bits, round to nearest even."""
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xf.shape, dtype=np.uint16)
    lib().orc_float_to_bf16(_p(xf), _p(out), xf.size)
    return out


def _bf16_value(bits: int) -> Decimal:
    """Exact value of a finite BF16 bit pattern; +-inf stands for +-2^128 (the
    point past which round-to-nearest overflows)."""
    mag = bits & 0x7FFF
    if mag == 0x7F80:
        v = Decimal(2 ** 128)                          # exact integer
    else:
        v = Decimal(float(np.array([mag << 16], dtype=np.uint32).view(np.float32)[0]))
    return v.copy_negate() if bits & 0x8000 else v    # exact (no context rounding)


def silu_mul_decimal(gb: int, ub: int, guess: int) -> int:
    """BF16_RNE(silu(g) * u) decided in 80-digit decimal arithmetic, for the
    finite non-zero g and u whose float64 product lies too close to a BF16
    rounding midpoint.  `guess` is the float64 result; the exact one is it or
    a neighbour in magnitude.  silu(g) = g / (1 + e^-g) for g > 0 and
    g e^g / (1 + e^g) for g < 0 (the same function).  If e^-g underflows even
    the decimal exponent range (g > ~2e18), the decimal value is g * u itself
    while the true product is strictly smaller in magnitude: a tie is then
    broken towards zero, and any other tie is an error (the product of a
    non-zero BF16 and silu(g) is never exactly a midpoint)."""
    from decimal import MAX_EMAX, MIN_EMIN
    g = _bf16_value(gb)
    u = _bf16_value(ub)
    with localcontext() as ctx:
        ctx.prec = 80
        ctx.Emin = MIN_EMIN
        ctx.Emax = MAX_EMAX
        if g > 0:
            s = g / (1 + (-g).exp())
        else:
            e = g.exp()
            s = g * e / (1 + e)
        x = s * u
        sign = guess & 0x8000
        cands = {guess}
        mag = guess & 0x7FFF
        if mag < 0x7F80:
            cands.add(sign | (mag + 1))
        if mag > 0:
            cands.add(sign | (mag - 1))
        dist = sorted((abs(_bf16_value(c) - x), c) for c in cands)
        if dist[0][0] == dist[1][0]:
            if g > 0 and s == g:            # e^-g underflowed: |silu(g) u| < |g u|
                return min(dist[0][1], dist[1][1], key=lambda c: c & 0x7FFF)
            raise AssertionError("exact BF16 tie for g=%r u=%r" % (g, u))
        return dist[0][1]


def _resolve_hard(gbits: np.ndarray, ubits: np.ndarray, y: np.ndarray, hard: np.ndarray):
    for i in hard:
        y.flat[i] = silu_mul_decimal(int(gbits.flat[i]), int(ubits.flat[i]), int(y.flat[i]))


def silu_mul_pairs(g_bits, u_bits) -> np.ndarray:
    """Elementwise BF16_RNE(silu(g) * u) for BF16 bit patterns (uint16 arrays of
    one shape); see silu_mul_bf16 for the definition."""
    g = np.ascontiguousarray(np.asarray(g_bits, dtype=np.uint16))
    u = np.ascontiguousarray(np.broadcast_to(np.asarray(u_bits, dtype=np.uint16), g.shape))
    y = np.empty(g.shape, dtype=np.uint16)
    cap = max(4096, g.size // 256)
    hard = np.empty(cap, dtype=np.int64)
    cnt = lib().orc_silu_mul_pairs(_p(g), _p(u), g.size, _p(y), _p(hard), cap, threads())
    if cnt > cap:
        hard = np.empty(cnt, dtype=np.int64)
        cnt = lib().orc_silu_mul_pairs(_p(g), _p(u), g.size, _p(y), _p(hard), cnt, threads())
    _resolve_hard(g, u, y, hard[:cnt])
    silu_mul_pairs.last_hard_count = int(cnt)
    return y


silu_mul_pairs.last_hard_count = 0


def silu_mul_bf16(h):
    """MoE glue between the expert GEMMs: h BF16 [m, 2*inter] = [gate | up]
    (the gate_up projection's output), y BF16 [m, inter].

    Definition (the pages fix no activation arithmetic; summary page, section
    3.4.1 names the expert layers fc1/fc2 as quantized): y = BF16_RNE(silu(g) * u)
    with silu(g) = g / (1 + e^-g), the real product rounded once to the
    nearest BF16 (ties to even).  Special values as the IEEE evaluation of
    g * sigma(g) * u: NaN in -> NaN, silu(+inf) = +inf, silu(-inf) = NaN,
    silu(+-0) = +-0, 0 * inf = NaN.  Computed in float64, with the rare
    products near a rounding midpoint decided in decimal."""
    import torch
    hb = _u16(h)
    m, two_i = hb.shape
    inter = two_i // 2
    y = np.empty((m, inter), dtype=np.uint16)
    cap = max(4096, y.size // 256)
    hard = np.empty(cap, dtype=np.int64)
    cnt = lib().orc_silu_mul_bf16(_p(hb), m, inter, two_i, _p(y), _p(hard), cap, threads())
    if cnt > cap:
        hard = np.empty(cnt, dtype=np.int64)
        cnt = lib().orc_silu_mul_bf16(_p(hb), m, inter, two_i, _p(y), _p(hard), cnt, threads())
    _resolve_hard(np.ascontiguousarray(hb[:, :inter]), np.ascontiguousarray(hb[:, inter:]), y,
                  hard[:cnt])
    silu_mul_bf16.last_hard_count = int(cnt)
    return torch.from_numpy(y.view(np.int16)).view(torch.bfloat16)


silu_mul_bf16.last_hard_count = 0


def silu_mul_quantize(h):
    """silu_mul_bf16 followed by 1x128-group quantization of y."""
    return quantize_act_groupwise(silu_mul_bf16(h))


def kv_calibrate(x):
    """Per-head scales fl32(amax/448) of a BF16 [rows, heads, head_dim] K or V tensor."""
    xb = _u16(x)
    rows, heads, hd = xb.shape
    s = np.zeros(heads, dtype=np.float32)
    lib().orc_kv_calibrate(_p(xb), rows, heads, hd, _p(s), threads())
    return s


def kv_quantize(x, scales):
    """E4M3 codes of a BF16 [rows, heads, head_dim] tensor under per-head scales."""
    xb = _u16(x)
    rows, heads, hd = xb.shape
    s = np.ascontiguousarray(np.asarray(scales, dtype=np.float32))
    assert s.shape == (heads,)
    q = np.zeros(xb.shape, dtype=np.uint8)
    lib().orc_kv_quantize(_p(xb), rows, heads, hd, _p(s), _p(q), threads())
    return q


# ------------------------------------------------------------------ GEMMs --

def _idx(v, n):
    if v is None:
        return np.arange(n, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(v, dtype=np.int64))


def gemm_w8a8(qa, sa, qw, sw, rows=None, cols=None):
    """float64 Y = A_deq W_deq^T on the selected rows/cols.

    qa uint8 [M, K], sa float32 [K/128, M], qw uint8 [N, K],
    sw float32 [ceil(N/128), K/128].  Returns (Y64 [nr, nc], absprod [nr, nc])
    where absprod = |A_deq| |W_deq|^T (the per-element error scale).
    """
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    assert K % 128 == 0 and qw.shape[1] == K
    assert sa.shape == (K // 128, M) and sw.shape == ((N + 127) // 128, K // 128)
    r, c = _idx(rows, M), _idx(cols, N)
    y = np.zeros((r.size, c.size), dtype=np.float64)
    ab = np.zeros_like(y)
    lib().orc_gemm_w8a8_sampled(_p(qa), _p(sa), _p(qw), _p(sw), M, N, K, _p(r), r.size,
                                _p(c), c.size, _p(y), _p(ab), threads())
    return y, ab


def grouped_gemm_w8a8(qa, sa, qw, sw, offsets, rows=None, cols=None):
    """Per-expert float64 GEMM: rows of segment e use expert e's weights.

    qw uint8 [E, N, K], sw float32 [E, N/128, K/128], offsets int32 [E+1].
    Rows outside all segments come back as NaN.
    """
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, K = qa.shape
    E, N, K2 = qw.shape
    assert K2 == K and off.shape == (E + 1,)
    r, c = _idx(rows, M), _idx(cols, N)
    y = np.zeros((r.size, c.size), dtype=np.float64)
    ab = np.zeros_like(y)
    lib().orc_grouped_gemm_w8a8_sampled(_p(qa), _p(sa), _p(qw), _p(sw), _p(off), E, M, N, K,
                                        _p(r), r.size, _p(c), c.size, _p(y), _p(ab),
                                        threads())
    return y, ab


def bf16_round(y64) -> np.ndarray:
    """BF16 (round-to-nearest-even) of fl32(Y64), returned widened to float32."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(y64, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float32).numpy()


# --------------------------------------------------------------------- TIS --

_F32_OVERFLOW = Decimal(2 ** 128)   # exact; RN overflows to inf at/after the midpoint below this


def _dec(f32: np.float32) -> Decimal:
    f = float(f32)
    if np.isinf(f):
        return _F32_OVERFLOW if f > 0 else -_F32_OVERFLOW
    return Decimal(f)  # exact


def exp_rn32_decimal(delta: np.float32) -> np.float32:
    """Correctly rounded binary32 e^delta, decided with a 60-digit decimal exp.

    e^delta is transcendental for delta != 0, so it never equals a rounding
    boundary; 60 significant digits separate it from every boundary by a wide
    margin.  Candidates are the float nearest the float64 estimate and its two
    neighbours.
    """
    d = np.float32(delta)
    if np.isnan(d):
        return np.float32(np.nan)
    with localcontext() as ctx:
        ctx.prec = 60
        v = Decimal(float(d)).exp()
        with np.errstate(over="ignore"):
            guess = np.float32(np.exp(np.float64(d)))
        cands = {guess,
                 np.nextafter(guess, np.float32(np.inf)),
                 np.nextafter(guess, np.float32(-np.inf))}
        cands = [c for c in cands if not (np.isinf(c) and c < 0) and not c < 0]
        best = min(cands, key=lambda c: (abs(_dec(c) - v), int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def tis_exp(logp_train, logp_rollout) -> np.ndarray:
    """RN32(e^(fl32(lt - lr))) per token (the unclipped importance weight)."""
    lt = np.ascontiguousarray(np.asarray(logp_train, dtype=np.float32))
    lr = np.ascontiguousarray(np.asarray(logp_rollout, dtype=np.float32))
    assert lt.shape == lr.shape
    n = lt.size
    e = np.empty(lt.shape, dtype=np.float32)
    cap = max(1024, n // 4096)
    hard = np.empty(cap, dtype=np.int64)
    cnt = lib().orc_tis_exp(_p(lt), _p(lr), n, _p(e), _p(hard), cap, threads())
    if cnt > cap:   # more boundary cases than expected: redo with room for all
        hard = np.empty(cnt, dtype=np.int64)
        cnt = lib().orc_tis_exp(_p(lt), _p(lr), n, _p(e), _p(hard), cnt, threads())
    ef = e.reshape(-1)
    ltf, lrf = lt.reshape(-1), lr.reshape(-1)
    for i in hard[:cnt]:
        ef[i] = exp_rn32_decimal(np.float32(ltf[i] - lrf[i]))
    tis_exp.last_hard_count = int(cnt)
    return e


tis_exp.last_hard_count = 0


def decode_attention_fp8kv(q, k_cache, v_cache, k_scale, v_scale, seq_lens, block_table=None,
                           page: int = None, sm_scale: float = None):
    """Decode attention over an FP8 E4M3 KV cache (summary page, section 3.4.4:
    the cache stores K and V in FP8 with per-head scales; the FP8 pipeline's
    attention reads them).  Plain float64 definition:

      K[t] = dec(k_code[t]) * k_scale[h],  V[t] = dec(v_code[t]) * v_scale[h]
      s_t  = sm_scale * <q, K[t]>,  p = softmax(s over t < len),  o = sum_t p_t V[t]

    for every sequence s and query head hq, with KV head h = hq // (Hq / Hkv)
    (grouped-query attention).  Token t of sequence s lives in page
    block_table[s, t // page] at slot t % page; with block_table None the cache
    is contiguous: page = its token dimension, sequence s in page s.
      q        BF16 (or float) [S, Hq, D]
      k_cache, v_cache  uint8 [pages, page, Hkv, D]
      seq_lens int [S]
    Returns float64 [S, Hq, D] (zeros for an empty context) and the float64
    sum_t p_t |V[t]| [S, Hq, D] (the scale of the result, for tolerances)."""
    import torch
    qf = (q.float().numpy() if isinstance(q, torch.Tensor) else np.asarray(q)).astype(np.float64)
    kc = np.asarray(k_cache, dtype=np.uint8)
    vc = np.asarray(v_cache, dtype=np.uint8)
    S, Hq, D = qf.shape
    npages, pg, Hkv, _ = kc.shape
    if page is None:
        page = pg
    group = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    ks = np.asarray(k_scale, dtype=np.float32).astype(np.float64)
    vs = np.asarray(v_scale, dtype=np.float32).astype(np.float64)
    dec = e4m3_decode(np.arange(256, dtype=np.uint8))
    out = np.zeros((S, Hq, D))
    mag = np.zeros((S, Hq, D))
    for si in range(S):
        n = int(seq_lens[si])
        if n <= 0:
            continue
        t = np.arange(n)
        pages = (np.asarray(block_table)[si, t // page] if block_table is not None
                 else np.full(n, si))
        slot = t % page
        for h in range(Hkv):
            K = dec[kc[pages, slot, h, :]] * ks[h]            # [n, D]
            V = dec[vc[pages, slot, h, :]] * vs[h]
            for hq in range(h * group, (h + 1) * group):
                sc = sm_scale * (K @ qf[si, hq])
                e = np.exp(sc - sc.max())
                p = e / e.sum()
                out[si, hq] = p @ V
                mag[si, hq] = p @ np.abs(V)
    return out, mag


IS_TRUNCATE, IS_MASK = 0, 1


def _sum64(x: np.ndarray) -> float:
    """Correctly rounded float64 sum of the given values (IEEE propagation of
    non-finite values)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    if not np.isfinite(x).all():
        return float(np.sum(x))
    return math.fsum(x.tolist())


def is_weights_stats(logp_train, logp_rollout, mask=None, c_hi: float = 2.0, c_lo: float = 0.0,
                     mode: int = IS_TRUNCATE, loss=None):
    """Importance weights of one batch with their mismatch statistics.

    Summary page, section 3.4.3: the weight w = pi_theta / pi_fp8 =
    exp(logp_train - logp_rollout); TIS truncates it at C, and the section names
    masked importance sampling (MIS) as the stronger alternative.  Section
    "Experimental setup / Metrics" (same page) tracks the mismatch KL
    D_KL(pi_fp8 || pi_theta) and, for end-to-end FP8, the sampling importance
    ratio.  Readings (the pages give no estimator):

    * mode IS_TRUNCATE: w as in tis_weights; IS_MASK: w = e if c_lo <= e <= c_hi,
      else 0 (NaN -> 0).  Masked-out tokens (mask == 0) get w = 0 either way.
    * over the valid tokens (mask != 0), with d = fl32(lt - lr), e = RN32(e^d):
      stats[0] = number of valid tokens,
      stats[1] = sum of fl32(lr - lt)           (k1: its mean estimates the KL,
                                                 tokens being drawn from pi_fp8),
      stats[2] = sum of fl32(fl32(e - 1) - d)   (k3 = (r - 1) - log r, r = e^d),
      stats[3] = sum of e                       (mean = sampling IS ratio),
      stats[4] = number of valid tokens whose weight was clipped (TIS) or
                 masked to 0 (MIS).
      Sums are returned (not means) so that batches can be combined.
    * with a per-token loss l (the trainer's policy-gradient loss of each
      token; section 3.4.3 multiplies it by the truncated weight in token-level
      TIS), stats[5] = sum over the valid tokens of fl32(w * l): the
      importance-weighted token loss (divide by stats[0] for its mean).
    """
    lt = np.asarray(logp_train, dtype=np.float32).reshape(-1)
    lr = np.asarray(logp_rollout, dtype=np.float32).reshape(-1)
    e = tis_exp(lt, lr).reshape(-1)
    d = (lt - lr).astype(np.float32)
    hi, lo = np.float32(c_hi), np.float32(c_lo)
    if mode == IS_TRUNCATE:
        w = np.where(e > hi, hi, e)
        changed = e > hi
        if c_lo > 0:
            w = np.where(e < lo, lo, w)
            changed = changed | (e < lo)
    elif mode == IS_MASK:
        keep = (e >= lo) & (e <= hi)
        w = np.where(keep, e, np.float32(0))
        changed = ~keep
    else:
        raise ValueError("mode must be IS_TRUNCATE or IS_MASK")
    valid = np.ones(lt.shape, dtype=bool) if mask is None else (np.asarray(mask).reshape(-1) != 0)
    w = np.where(valid, w, np.float32(0)).astype(np.float32)
    k1 = (lr - lt).astype(np.float32)
    k3 = ((e - np.float32(1)).astype(np.float32) - d).astype(np.float32)
    stats = np.array([float(valid.sum()), _sum64(k1[valid]), _sum64(k3[valid]), _sum64(e[valid]),
                      float((changed & valid).sum())], dtype=np.float64)
    terms_abs = np.array([0.0, _sum64(np.abs(k1[valid])), _sum64(np.abs(k3[valid])),
                          _sum64(np.abs(e[valid])), 0.0])
    if loss is not None:
        lw = (w * np.asarray(loss, dtype=np.float32).reshape(-1)).astype(np.float32)
        stats = np.append(stats, _sum64(lw[valid]))
        terms_abs = np.append(terms_abs, _sum64(np.abs(lw[valid])))
    return w, stats, terms_abs


def tis_weights(logp_train, logp_rollout, mask=None, c_hi: float = 2.0, c_lo: float = 0.0):
    """Token-level truncated importance weights.

    Summary page, section 3.4.3: w = pi_theta / pi_fp8 = exp(logp_train -
    logp_rollout), truncated at C = 2.  One-sided min(w, C) by default
    (c_lo = 0); c_lo = 1/C gives the two-sided [1/C, C] clip the same section
    also states.  Comparisons act on the rounded weight; NaN stays NaN; tokens
    with mask == 0 get weight 0.
    """
    e = tis_exp(logp_train, logp_rollout)
    hi, lo = np.float32(c_hi), np.float32(c_lo)
    w = np.where(e > hi, hi, e)
    if c_lo > 0:
        w = np.where(e < lo, lo, w)
    if mask is not None:
        w = np.where(np.asarray(mask) == 0, np.float32(0), w)
    return w.astype(np.float32)
