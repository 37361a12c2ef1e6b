"""The allocation-free KV calibration entry point, called through the C ABI.

fp8rl_quantize_kv_fp8_calibrate_noalloc serves callers that cannot let the
library allocate device memory (for example an engine that hands almost all
of the GPU's memory to its own pools up front).  Its results must be
identical to the ordinary fp8rl_quantize_kv_fp8(..., FP8RL_KV_CALIBRATE, ...)
call, and both must equal the oracle's KV calibration and quantization bit
for bit.  Two calls in a row check that the shared scratch array is cleared
between calls: the first input has much larger maxima than the second, so
stale maxima would show up as wrong scales.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_rollout_gb300 import binding, workloads
from gpu_helpers import device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _lib():
    L = binding.load()
    fn = L.fp8rl_quantize_kv_fp8_calibrate_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P, P]
    return L


def _reference(L, x, heads, hd, stream):
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty(heads, dtype=torch.float32, device=x.device)
    st = L.fp8rl_quantize_kv_fp8(x.data_ptr(), x.numel() // (heads * hd), heads, hd,
                                 binding.FP8RL_KV_CALIBRATE, s.data_ptr(), q.data_ptr(), stream)
    assert st == 0, binding.last_error()
    return q, s


def test_noalloc_matches_calibrate_on_two_calls_in_a_row():
    dev = device()
    L = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    heads, hd = 8, 128
    big = workloads.kv_tensor(seed=41, device=dev, seqs=2, tokens=300, heads=heads, head_dim=hd)
    big = (big.float() * 30.0).to(torch.bfloat16)
    small = workloads.kv_tensor(seed=42, device=dev, seqs=3, tokens=77, heads=heads, head_dim=hd)
    for x in (big, small):
        q = torch.full(x.shape, 0x5A, dtype=torch.uint8, device=dev)
        s = torch.full((heads,), -1.0, dtype=torch.float32, device=dev)
        st = L.fp8rl_quantize_kv_fp8_calibrate_noalloc(x.data_ptr(), x.numel() // (heads * hd),
                                                       heads, hd, s.data_ptr(), q.data_ptr(),
                                                       stream)
        assert st == 0, binding.last_error()
        qr, sr = _reference(L, x, heads, hd, stream)
        torch.cuda.synchronize()
        assert (np_f32_bits(s) == np_f32_bits(sr)).all()
        assert (np_u8(q) == np_u8(qr)).all()
        # and directly against the oracle
        xr = x.view(-1, heads, hd).cpu()
        os_ = oracle.kv_calibrate(xr)
        assert (np_f32_bits(s) == os_.view(np.uint32)).all()
        assert (np_u8(q).reshape(-1, heads, hd) == oracle.kv_quantize(xr, os_)).all()


def test_noalloc_rejects_more_heads_than_its_scratch_holds():
    device()
    L = _lib()
    fake = 1 << 20          # never dereferenced: the call fails its checks first
    st = L.fp8rl_quantize_kv_fp8_calibrate_noalloc(fake, 4, 257, 8, fake, fake, None)
    assert st == 3
    assert "at most 256 heads" in binding.last_error()
