"""Pins of the oracle's FP8-KV decode attention, against things other than itself:

* torch's scaled_dot_product_attention in float64 on the dequantized cache
  (a library routine), with grouped-query heads expanded and ragged lengths;
* closed forms: one token returns its value row; equal keys average the values;
* a paged cache (shuffled pages + block table) equals the contiguous one;
* query head hq reads KV head hq // (Hq / Hkv) and no other.
"""
import math

import numpy as np
import torch

import oracle


def _cache(rng, pages, page, hkv, d):
    kc = rng.integers(0, 256, size=(pages, page, hkv, d)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(pages, page, hkv, d)).astype(np.uint8)
    for c in (kc, vc):
        c[(c & 0x7F) == 0x7F] = 0x3C            # no NaN codes
    return kc, vc


def test_matches_torch_sdpa_float64():
    rng = np.random.default_rng(0)
    S, Hq, Hkv, D, T = 3, 8, 2, 128, 70
    kc, vc = _cache(rng, S, T, Hkv, D)
    ks = np.array([0.013, 0.021], np.float32)
    vs = np.array([0.11, 0.07], np.float32)
    q = torch.randn(S, Hq, D).to(torch.bfloat16)
    lens = [70, 1, 33]
    out, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, lens)
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    for s in range(S):
        n = lens[s]
        K = torch.from_numpy(dec[kc[s, :n]] * ks.astype(np.float64)[None, :, None])   # [n, Hkv, D]
        V = torch.from_numpy(dec[vc[s, :n]] * vs.astype(np.float64)[None, :, None])
        K = K.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)                     # [Hq, n, D]
        V = V.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        qq = q[s].double().unsqueeze(1)                                                 # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, K, V).squeeze(1).numpy()
        assert np.allclose(out[s], ref, rtol=1e-12, atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(1)
    kc, vc = _cache(rng, 2, 16, 1, 128)
    ks, vs = np.array([0.05], np.float32), np.array([0.2], np.float32)
    q = torch.randn(2, 4, 128).to(torch.bfloat16)
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    out, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, [1, 0])
    for hq in range(4):
        assert (out[0, hq] == dec[vc[0, 0, 0]] * np.float64(np.float32(0.2))).all()   # one token
    assert (out[1] == 0).all()                                                         # empty
    kc[1, :, 0, :] = kc[1, 0, 0, :]                                                    # equal keys
    out, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, [1, 16])
    want = (dec[vc[1, :, 0]] * np.float64(np.float32(0.2))).mean(axis=0)
    for hq in range(4):
        assert np.allclose(out[1, hq], want, rtol=1e-12, atol=1e-15)


def test_paged_equals_contiguous():
    rng = np.random.default_rng(2)
    S, T, page, Hkv, D = 3, 96, 32, 2, 128
    kc, vc = _cache(rng, S, T, Hkv, D)
    ks, vs = np.array([0.02, 0.03], np.float32), np.array([0.1, 0.05], np.float32)
    q = torch.randn(S, 4, D).to(torch.bfloat16)
    lens = [96, 50, 33]
    ref, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, lens)
    # split every sequence into 3 pages of 32 tokens and scatter them in a shuffled pool
    perm = rng.permutation(S * 3)
    kp = np.zeros((S * 3 + 2, page, Hkv, D), np.uint8)
    vp = np.zeros_like(kp)
    table = np.zeros((S, 3), np.int32)
    for s in range(S):
        for j in range(3):
            dst = perm[s * 3 + j] + 2
            kp[dst] = kc[s, j * page:(j + 1) * page]
            vp[dst] = vc[s, j * page:(j + 1) * page]
            table[s, j] = dst
    out, _ = oracle.decode_attention_fp8kv(q, kp, vp, ks, vs, lens, block_table=table, page=page)
    assert (out == ref).all()


def test_query_head_reads_its_kv_group_only():
    rng = np.random.default_rng(3)
    kc, vc = _cache(rng, 1, 20, 4, 128)
    ks, vs = np.full(4, 0.02, np.float32), np.full(4, 0.1, np.float32)
    q = torch.randn(1, 8, 128).to(torch.bfloat16)
    base, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, [20])
    vc2 = vc.copy()
    vc2[:, :, 2, :] = 0                                      # KV head 2 -> query heads 4, 5
    out, _ = oracle.decode_attention_fp8kv(q, kc, vc2, ks, vs, [20])
    assert (out[0, 4:6] == 0).all()
    assert (out[0, :4] == base[0, :4]).all() and (out[0, 6:] == base[0, 6:]).all()
    sm = 1.0 / math.sqrt(128)
    out2, _ = oracle.decode_attention_fp8kv(q, kc, vc, ks, vs, [20], sm_scale=sm)
    assert (out2 == base).all()
