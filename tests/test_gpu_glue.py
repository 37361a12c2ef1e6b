"""GPU parity of the MoE glue against the oracle, bit-exact: the gather +
1x128 quantization of expert-sorted rows, and the SiLU(gate) * up +
quantization between the expert GEMMs, on the Qwen3-30B-A3B routing at full
size, ragged shapes, strided inputs, special values, and out-of-range
gather indices (reported, not faulted).  The gated activation itself,
y = BF16_RNE(silu(g) * u), is compared over every BF16 gate with every up
significand (both signs) and with every up exponent: the rounding of the
product depends only on the two significands except where it overflows or
turns subnormal, which the exponent sweep covers."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import Canary, device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _gather_case(a_cpu, rows_np, dev, lda_pad=0):
    m_src, k = a_cpu.shape
    if lda_pad:
        big = torch.zeros(m_src, k + lda_pad, dtype=torch.bfloat16, device=dev)
        big[:, :k] = a_cpu.to(dev)
        a = big[:, :k]
    else:
        a = a_cpu.to(dev)
    m = len(rows_np)
    qc = Canary(m * k, torch.uint8, dev)
    sc = Canary(((k + 127) // 128) * m, torch.float32, dev)
    rows = torch.from_numpy(np.asarray(rows_np, dtype=np.int32)).to(dev)
    q, s = fp8rl.quantize_act_gather(a, rows, qc.view.view(m, k), sc.view.view((k + 127) // 128, m))
    torch.cuda.synchronize()
    qc.check(); sc.check()
    fp8rl.device_status(0)
    oq, os_ = oracle.quantize_act_gather(a_cpu, rows_np)
    assert (np_u8(q) == oq).all()
    assert (np_f32_bits(s) == os_.view(np.uint32)).all()


def test_gather_moe_routing_full():
    dev = device()
    _, token_of_row, _ = workloads.moe_routing(seed=0)
    x = workloads.dense_acts(workloads.MOE_TOKENS, workloads.MOE_HIDDEN, seed=8)
    _gather_case(x, token_of_row.numpy(), dev)


@pytest.mark.parametrize("m_src,k,m", [(5, 8, 9), (40, 200, 17), (300, 768, 1000), (7, 1032, 3)])
def test_gather_ragged_shapes(m_src, k, m):
    dev = device()
    rows = np.random.default_rng(m).integers(0, m_src, size=m)
    _gather_case(workloads.dense_acts(m_src, k, seed=k), rows, dev)


def test_gather_row_stride():
    dev = device()
    _gather_case(workloads.dense_acts(33, 640, seed=3), np.array([32, 0, 5, 5, 17]), dev, lda_pad=24)


def test_gather_out_of_range_index_is_reported():
    dev = device()
    a = workloads.dense_acts(10, 256, seed=5).to(dev)
    rows = torch.tensor([3, -1, 10, 9], dtype=torch.int32, device=dev)
    q, s = fp8rl.quantize_act_gather(a, rows)
    with pytest.raises(fp8rl.Fp8rlError) as ei:
        fp8rl.device_status(0)
    assert "out of range" in str(ei.value)
    fp8rl.device_status(0)                      # cleared by the failing read
    qn, sn = np_u8(q), s.cpu().numpy()
    assert (qn[1] == 0).all() and (qn[2] == 0).all() and (sn[:, 1] == 0).all() and (sn[:, 2] == 0).all()
    oq, os_ = oracle.quantize_act_gather(a.cpu(), [3, 9])
    assert (qn[[0, 3]] == oq).all() and (sn[:, [0, 3]] == os_).all()


def _silu_case(h_cpu, dev, ld_pad=0):
    m, two_i = h_cpu.shape
    inter = two_i // 2
    if ld_pad:
        big = torch.zeros(m, two_i + ld_pad, dtype=torch.bfloat16, device=dev)
        big[:, :two_i] = h_cpu.to(dev)
        h = big[:, :two_i]
    else:
        h = h_cpu.to(dev)
    qc = Canary(m * inter, torch.uint8, dev)
    sc = Canary(((inter + 127) // 128) * m, torch.float32, dev)
    q, s = fp8rl.silu_mul_quantize(h, qc.view.view(m, inter),
                                   sc.view.view((inter + 127) // 128, m))
    torch.cuda.synchronize()
    qc.check(); sc.check()
    oq, os_ = oracle.silu_mul_quantize(h_cpu)
    assert (np_f32_bits(s) == os_.view(np.uint32)).all()
    bad = np_u8(q) != oq
    assert not bad.any(), "codes differ at %s" % np.argwhere(bad)[:5].ravel()


def test_silu_moe_gate_up_output_full():
    """The gate_up projection's output for 32768 routed rows (N(0,1)-scaled
    like the product of N(0,1) inputs and N(0, 0.02) weights over K = 2048)."""
    dev = device()
    rows = workloads.MOE_TOKENS * workloads.MOE_TOPK
    h = workloads.expert_inputs(rows, 2 * workloads.MOE_INTER, seed=11).float().mul_(0.9)
    _silu_case(h.to(torch.bfloat16), dev)


@pytest.mark.parametrize("m,inter", [(1, 8), (3, 200), (17, 768), (130, 1032)])
def test_silu_ragged_shapes(m, inter):
    dev = device()
    _silu_case(workloads.expert_inputs(m, 2 * inter, seed=m + inter), dev)


def test_silu_row_stride_and_special_values():
    dev = device()
    rng = np.random.default_rng(12)
    g = rng.normal(0, 6, size=(40, 256)).astype(np.float32)
    g[0, :16] = [0.0, -0.0, -88.5, -100.0, -87.9, 87.0, 88.5, 1e-30, -1e-30, 3e4, -3e4, 15.0,
                 -15.0, 0.5, -0.5, 2.0 ** -130]
    u = rng.normal(0, 2, size=(40, 256)).astype(np.float32)
    u[1] = 0.0
    u[2, ::3] = -0.0
    h = torch.from_numpy(np.concatenate([g, u], axis=1)).to(torch.bfloat16)
    _silu_case(h, dev)
    _silu_case(h, dev, ld_pad=16)


def test_silu_every_bf16_gate():
    """All 65536 BF16 gate bit patterns (NaN, infinities, subnormals, both
    zeros) against the oracle, each with three up values: the activation is a
    function of the gate alone, so this covers every value it can take."""
    dev = device()
    gates = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    g = gates.view(512, 128)
    rng = np.random.default_rng(13)
    for up in (torch.ones(512, 128), torch.from_numpy(rng.normal(0, 3, (512, 128)).astype(np.float32)),
               torch.full((512, 128), -1e-3)):
        h = torch.cat([g, up.to(torch.bfloat16)], dim=1)
        _silu_case(h, dev)


def _pairs_case(dev, g_bits: np.ndarray, u_rows: np.ndarray):
    """One row per up value: h[r] = [all gates | u_rows[r] repeated]; y from the
    library's BF16 entry against the oracle's pairs, bit for bit."""
    rows, inter = u_rows.size, g_bits.size
    h = np.empty((rows, 2 * inter), dtype=np.uint16)
    h[:, :inter] = g_bits[None, :]
    h[:, inter:] = u_rows[:, None]
    ht = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    yc = Canary(rows * inter, torch.bfloat16, dev)
    y = fp8rl.silu_mul_bf16(ht, yc.view.view(rows, inter))
    torch.cuda.synchronize()
    yc.check()
    got = y.cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    want = oracle.silu_mul_pairs(np.tile(g_bits, rows), np.repeat(u_rows, inter))
    bad = got != want
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError("y differs: g=%s u=%s gpu=%s oracle=%s" % (
            [hex(x) for x in np.tile(g_bits, rows)[i]], [hex(x) for x in np.repeat(u_rows, inter)[i]],
            [hex(x) for x in got[i]], [hex(x) for x in want[i]]))


def test_silu_mul_bf16_every_gate_every_up_significand():
    """All 65536 gates x all 256 up significands of [1, 2), both signs (2^25 products)."""
    dev = device()
    g = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for sign in (0x0000, 0x8000):
        _pairs_case(dev, g, (sign | 0x3F80 | np.arange(128)).astype(np.uint16))
        _pairs_case(dev, g, (sign | 0x4000 | np.arange(128)).astype(np.uint16))   # [2, 4): odd exponent


def test_silu_mul_bf16_every_gate_every_up_exponent():
    """All gates x every up exponent field (zeros, subnormals, infinities and
    NaNs included) with three significands and both signs: overflow to inf,
    subnormal and zero results, and the special values."""
    dev = device()
    g = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for mant in (0x00, 0x5B, 0x7F):
        for sign in (0x0000, 0x8000):
            _pairs_case(dev, g, (sign | (np.arange(256) << 7) | mant).astype(np.uint16))


def test_silu_mul_bf16_strided_and_random():
    dev = device()
    rng = np.random.default_rng(21)
    m, inter = 37, 392
    h = rng.integers(0, 1 << 16, size=(m, 2 * inter + 24)).astype(np.uint16)
    ht = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)[:, :2 * inter]
    ybig = torch.zeros(m, inter + 40, dtype=torch.bfloat16, device=dev)
    fp8rl.silu_mul_bf16(ht, ybig[:, :inter])
    torch.cuda.synchronize()
    got = ybig.cpu().view(torch.int16).numpy().view(np.uint16)
    want = oracle.silu_mul_bf16(torch.from_numpy(np.ascontiguousarray(h[:, :2 * inter]).view(np.int16))
                                .view(torch.bfloat16)).view(torch.int16).numpy().view(np.uint16)
    assert (got[:, :inter] == want).all()
    assert (got[:, inter:] == 0).all()


def test_silu_quantize_equals_quantized_bf16_glue():
    """The fused glue equals the BF16 glue followed by the activation quantizer."""
    dev = device()
    h = workloads.expert_inputs(300, 2 * 768, seed=22).to(dev)
    q1, s1 = fp8rl.silu_mul_quantize(h)
    q2, s2 = fp8rl.quantize_act_groupwise(fp8rl.silu_mul_bf16(h))
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1.view(torch.int32), s2.view(torch.int32))
