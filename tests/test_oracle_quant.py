"""Pins of the oracle's quantizers (weights 128x128, activations 1x128, KV).

Checked against hand-worked groups (golden/quant_worked_examples.json), the
invariants the pages' definition implies (the block max maps onto +-448; every
element is within half an E4M3 step of x/scale), the layout of each scale set,
and cross-consistency between the three quantizers (one definition, three
tilings).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_rollout_gb300 import workloads


def _bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    assert (t.to(torch.float32) == torch.tensor(values, dtype=torch.float32)).all(), \
        "worked example values must be exact in bf16"
    return t


def test_worked_groups(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "quant_worked_examples.json")))
    for grp in g["groups"]:
        vals = grp["values"]
        row = torch.zeros(1, 128, dtype=torch.bfloat16)
        row[0, :len(vals)] = _bf16_bits(vals)
        q, s = oracle.quantize_act_groupwise(row)
        assert hex(int(s.view(np.uint32)[0, 0])) == hex(int(grp["scale_hex"], 16)), grp["name"]
        want = [int(c, 16) for c in grp["codes"]]
        assert list(q[0, :len(vals)]) == want, grp["name"]
        assert (q[0, len(vals):] == 0).all()


def test_block_max_maps_to_448_and_error_bound():
    w = workloads.make_weight(384, 640, seed=3)
    q, s = oracle.quantize_weights_blockwise(w)
    wf = w.to(torch.float64).numpy()
    deq = oracle.e4m3_decode(q)
    for bi in range(s.shape[0]):
        for bj in range(s.shape[1]):
            blk = np.s_[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            codes = q[blk]
            assert ((codes & 0x7F) == 0x7E).any()            # the max element lands on 448
            assert ((codes & 0x7F) <= 0x7E).all()
            sc = np.float64(s[bi, bj])
            x = wf[blk] / sc                                  # real quotient
            d = deq[blk]
            # within half a grid step (relative 1/16 for normals, 2^-10 absolute below),
            # plus the binary32 rounding of the quotient
            bound = np.maximum(np.abs(x) / 16.0, 2.0 ** -10) * (1 + 2.0 ** -20) + 448 * 2.0 ** -23
            assert (np.abs(d - x) <= bound).all()


def test_weight_blocks_ignore_out_of_range_elements():
    """A ragged edge block takes its max over valid elements only: padding
    the matrix with a huge column outside the block must not move the scale."""
    w = workloads.make_weight(130, 200, seed=4)
    q, s = oracle.quantize_weights_blockwise(w)
    assert s.shape == (2, 2)
    # same top-left 128x128 block embedded in a bigger matrix with a spike outside it
    big = torch.zeros(256, 256, dtype=torch.bfloat16)
    big[:130, :200] = w
    big[129, 130] = 1000.0            # row 129 is in block row 1, col 130 in block col 1
    q2, s2 = oracle.quantize_weights_blockwise(big)
    assert s2[0, 0] == s[0, 0] and s2[0, 1] == s[0, 1] and s2[1, 0] == s[1, 0]
    assert s2[1, 1] == np.float32(1000.0) / np.float32(448.0)
    assert (q2[:128, :128] == q[:128, :128]).all()
    # and a block of 2 valid rows x 72 valid cols has the max of exactly those
    blk = w[128:130, 128:200].to(torch.float32).abs().max().item()
    assert s[1, 1] == np.float32(blk) / np.float32(448.0)


def test_one_row_weight_equals_activation_group():
    """A [1, K] weight has 1x128 blocks: both tilings must agree exactly."""
    a = workloads.dense_acts(1, 1024, seed=5)
    qw, sw = oracle.quantize_weights_blockwise(a)
    qa, sa = oracle.quantize_act_groupwise(a)
    assert (qw == qa).all()
    assert (sw[0] == sa[:, 0]).all()


def test_act_scale_layout_is_group_major():
    a = workloads.dense_acts(5, 384, seed=6)
    q, s = oracle.quantize_act_groupwise(a)
    assert s.shape == (3, 5)
    af = a.to(torch.float32).numpy()
    for r in range(5):
        for gi in range(3):
            amax = np.abs(af[r, gi * 128:(gi + 1) * 128]).max()
            assert s[gi, r] == np.float32(amax) / np.float32(448.0)
    # the codes of each group equal the element map under that group's scale
    for r in range(5):
        for gi in range(3):
            x = af[r, gi * 128:(gi + 1) * 128]
            assert (q[r, gi * 128:(gi + 1) * 128] == oracle.quantize_values(x, s[gi, r])).all()


def test_act_ragged_last_group():
    a = workloads.dense_acts(3, 200, seed=7)
    q, s = oracle.quantize_act_groupwise(a)
    af = a.to(torch.float32).numpy()
    assert s.shape == (2, 3)
    for r in range(3):
        assert s[1, r] == np.float32(np.abs(af[r, 128:200]).max()) / np.float32(448.0)


def test_kv_per_head_scales_and_codes():
    x = workloads.kv_tensor(seed=8, seqs=2, tokens=37, heads=4, head_dim=64)
    xr = x.view(-1, 4, 64)
    s = oracle.kv_calibrate(xr)
    xf = xr.to(torch.float32).numpy()
    for h in range(4):
        assert s[h] == np.float32(np.abs(xf[:, h, :]).max()) / np.float32(448.0)
    q = oracle.kv_quantize(xr, s)
    for h in range(4):
        assert (q[:, h, :] == oracle.quantize_values(xf[:, h, :], s[h])).all()
        assert ((q[:, h, :] & 0x7F) == 0x7E).any()
    # a head quantized with the per-head scale equals a 1-row "weight" with that scale:
    # one definition of the element map across all three quantizers
    row = xr[:, 1, :].reshape(1, -1)[:, :128]
    qa, sa = oracle.quantize_act_groupwise(row)
    assert (oracle.quantize_values(row.to(torch.float32).numpy(), sa[0, 0]) == qa).all()


def test_element_map_division_not_reciprocal_multiply():
    """The reading is x / s in binary32, not x * (1/s): find inputs where the
    two differ and check the oracle follows the division."""
    rng = np.random.default_rng(9)
    amax = np.float32(rng.uniform(1e-3, 10))
    s = np.float32(amax) / np.float32(448)
    x = rng.uniform(-float(amax), float(amax), 200000).astype(np.float32)
    by_div = (x / s).astype(np.float32)
    by_mul = (x * (np.float32(1) / s)).astype(np.float32)
    diff = by_div != by_mul
    assert diff.any()
    want = oracle.e4m3_encode(by_div)
    assert (oracle.quantize_values(x, s) == want).all()
