"""The C-ABI library: it loads, exports every symbol include/fp8rl.h declares,
and rejects bad arguments on the host before touching a GPU (no compute
calls here; this file runs on machines without a GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from fp8_precision_rollout_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load()


def _exported_fp8rl_symbols():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    return sorted(set(re.findall(r"\b(fp8rl_[a-z0-9_]+)\b", out)))


def test_exports_every_declared_symbol(lib):
    declared = binding.declared_symbols()
    assert len(declared) >= 18
    # the library's exported C symbols are exactly the header's declarations
    assert _exported_fp8rl_symbols() == declared
    for name in declared:
        assert hasattr(lib, name), name
    # and the binding wraps each of them under the same name
    for name in declared:
        if name in ("fp8rl_last_error", "fp8rl_version", "fp8rl_device_status"):
            continue
        assert hasattr(binding, name[len("fp8rl_"):]), name


def test_version(lib):
    hdr = open(binding.HEADER).read()
    want = int(re.search(r"#define FP8RL_VERSION (\d+)", hdr).group(1))
    assert binding.version() == want


NULL = None


def test_host_validation_before_any_launch(lib):
    # null pointers
    assert lib.fp8rl_quantize_act_groupwise(NULL, 4, 128, 128, NULL, NULL, NULL) == 1
    assert lib.fp8rl_tis_weights(NULL, NULL, NULL, 4, 2.0, 0.0, NULL, NULL) == 1
    assert lib.fp8rl_gemm_w8a8_blockwise(NULL, NULL, NULL, NULL, 1, 256, 128, NULL, 256, NULL) == 1
    assert "null" in binding.last_error()
    fake = 1 << 20   # aligned, never dereferenced: every call below fails its checks first
    # k not a multiple of 8 -> alignment
    assert lib.fp8rl_quantize_act_groupwise(fake, 4, 100, 100, fake, fake, NULL) == 2
    # misaligned pointer
    assert lib.fp8rl_quantize_act_groupwise(fake + 2, 4, 128, 128, fake, fake, NULL) == 2
    # lda < k
    assert lib.fp8rl_quantize_act_groupwise(fake, 4, 128, 64, fake, fake, NULL) == 1
    # GEMM: k % 128, n % 16, ldy
    assert lib.fp8rl_gemm_w8a8_blockwise(fake, fake, fake, fake, 8, 256, 100, fake, 256, NULL) == 3
    assert lib.fp8rl_gemm_w8a8_blockwise(fake, fake, fake, fake, 8, 250, 128, fake, 256, NULL) == 3
    assert lib.fp8rl_gemm_w8a8_blockwise(fake, fake, fake, fake, 8, 256, 128, fake, 200, NULL) == 2
    assert lib.fp8rl_gemm_w8a8_blockwise(fake, fake, fake, fake, -1, 256, 128, fake, 256, NULL) == 1
    # grouped: experts range, n % 128
    assert lib.fp8rl_grouped_gemm_w8a8_blockwise(fake, fake, fake, fake, fake, 0, 8, 256, 128,
                                                 fake, NULL) == 3
    assert lib.fp8rl_grouped_gemm_w8a8_blockwise(fake, fake, fake, fake, fake, 2000, 8, 256, 128,
                                                 fake, NULL) == 3
    assert lib.fp8rl_grouped_gemm_w8a8_blockwise(fake, fake, fake, fake, fake, 4, 8, 200, 128,
                                                 fake, NULL) == 3
    # KV: mode, head_dim % 8, heads*hd limit
    assert lib.fp8rl_quantize_kv_fp8(fake, 4, 8, 128, 7, fake, fake, NULL) == 1
    assert lib.fp8rl_quantize_kv_fp8(fake, 4, 8, 100, 0, fake, fake, NULL) == 2
    assert lib.fp8rl_quantize_kv_fp8(fake, 4, 32, 128, 0, fake, fake, NULL) == 3
    # TIS: clip bounds
    assert lib.fp8rl_tis_weights(fake, fake, NULL, 4, 0.0, 0.0, fake, NULL) == 1
    assert lib.fp8rl_tis_weights(fake, fake, NULL, 4, 2.0, 3.0, fake, NULL) == 1
    assert lib.fp8rl_tis_weights(fake, fake, NULL, 4, float("inf"), 0.0, fake, NULL) == 1
    assert lib.fp8rl_tis_weights(fake, fake, NULL, -1, 2.0, 0.0, fake, NULL) == 1
    # weights: descriptor checks, including a bad tensor inside a batch
    good = binding.WDesc(fake, fake, fake, 128, 128, 128, 128)
    bad = binding.WDesc(fake, fake, fake, 128, 100, 104, 104)
    arr = (binding.WDesc * 2)(good, bad)
    assert lib.fp8rl_quantize_weights_blockwise_multi(ctypes.addressof(arr), 2, NULL) == 2
    assert "tensor 1" in binding.last_error()
    assert lib.fp8rl_quantize_weights_blockwise_multi(NULL, 3, NULL) == 1
    assert lib.fp8rl_quantize_weights_blockwise(fake, 0, 128, 128, fake, 128, fake, NULL) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="libfp8rl.so not found"):
        binding.load(str(tmp_path / "missing" / "libfp8rl.so"))


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.dirname(binding.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "fp8rl_oracle" not in text, f


def test_error_path_entries_check_their_arguments_on_the_host(lib):
    assert lib.fp8rl_inject_device_status(0, 4, 0) == 1            # unknown flag
    assert "unknown status flags" in binding.last_error()
    assert lib.fp8rl_selftest_bounded_wait(0, None) == 1            # limit out of range
    assert lib.fp8rl_selftest_bounded_wait(1000001, None) == 1


def test_decode_linear_checks_shapes_on_the_host(lib):
    fake = 1 << 20          # never dereferenced: the call fails its checks first
    f = lib.fp8rl_linear_w8a8_decode
    # m > 256
    assert f(fake, 128, fake, fake, fake, fake, 257, 128, 128, fake, 128, 1 << 12, 1 << 30, None) == 3
    # n not a multiple of 128
    assert f(fake, 128, fake, fake, fake, fake, 16, 200, 128, fake, 200, 1 << 12, 1 << 30, None) == 3
    # null workspace
    assert f(fake, 128, fake, fake, fake, fake, 16, 128, 128, fake, 128, None, 1 << 30, None) == 1
    # misaligned workspace
    assert f(fake, 128, fake, fake, fake, fake, 16, 128, 128, fake, 128, (1 << 12) + 16, 1 << 30,
             None) == 2
