"""The error path of the device status word, exercised without faulting the
GPU.  A host-injected status word must be reported by fp8rl_device_status
as the matching error (with the recorded site) and cleared by the read; a
kernel whose barrier wait runs out (the self-test kernel waits, with a 2 ms
limit, on a barrier nothing completes) must return and report
FP8RL_ERR_TIMEOUT, after which the context still computes correct results."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu

TIMEOUT, INVALID_ARG = 5, 1


def test_injected_timeout_is_reported_with_its_site_and_cleared():
    device()
    fp8rl.device_status(0)
    fp8rl.inject_device_status(0, 1, 31)
    with pytest.raises(fp8rl.Fp8rlError) as ei:
        fp8rl.device_status(0)
    assert ei.value.status == TIMEOUT and "site 31" in str(ei.value)
    fp8rl.device_status(0)                    # the failing read cleared it


def test_injected_bad_index_is_reported():
    device()
    fp8rl.inject_device_status(0, 2, 0)
    with pytest.raises(fp8rl.Fp8rlError) as ei:
        fp8rl.device_status(0)
    assert ei.value.status == INVALID_ARG and "out of range" in str(ei.value)
    fp8rl.device_status(0)


def test_status_read_without_clear_keeps_the_word():
    device()
    fp8rl.inject_device_status(0, 1, 7)
    for _ in range(2):
        with pytest.raises(fp8rl.Fp8rlError):
            fp8rl.device_status(0, clear=False)
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.device_status(0, clear=True)
    fp8rl.device_status(0)


def test_bounded_wait_times_out_and_the_context_survives():
    dev = device()
    fp8rl.device_status(0)
    fp8rl.selftest_bounded_wait(2000)
    torch.cuda.synchronize()                  # the kernel returned
    with pytest.raises(fp8rl.Fp8rlError) as ei:
        fp8rl.device_status(0)
    assert ei.value.status == TIMEOUT and "site 90" in str(ei.value)
    fp8rl.device_status(0)
    # the context still runs the library's kernels correctly
    a = workloads.dense_acts(64, 512, seed=3)
    q, s = fp8rl.quantize_act_groupwise(a.to(dev))
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    oq, os_ = oracle.quantize_act_groupwise(a)
    assert (np_u8(q) == oq).all() and (np_f32_bits(s) == os_.view(np.uint32)).all()
