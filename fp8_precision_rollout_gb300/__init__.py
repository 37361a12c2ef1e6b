"""GB300-native hot path of the FP8 RL rollout stack (FP8-RL, arXiv 2601.18150).

The compute lives in a C-ABI CUDA library (``libfp8rl.so``, sources in
``csrc/``, declarations in ``include/fp8rl.h``); :mod:`.binding` is a thin
ctypes layer with the same call names.  The library is loaded on the first
call and a missing or unloadable library raises -- there is no fallback.
"""
from .binding import (  # noqa: F401
    FP8RL_IS_MASK,
    FP8RL_IS_TRUNCATE,
    FP8RL_KV_CALIBRATE,
    FP8RL_KV_GIVEN,
    Fp8rlError,
    decode_attention_fp8kv,
    device_status,
    gemm_w8a8_blockwise,
    inject_device_status,
    grouped_gemm_w8a8_blockwise,
    is_weights_stats,
    is_weights_stats_loss,
    last_error,
    linear_w8a8_decode,
    linear_w8a8_decode_workspace_bytes,
    quantize_act_gather,
    quantize_act_groupwise,
    quantize_kv_fp8,
    quantize_weights_blockwise,
    quantize_weights_blockwise_multi,
    quantize_weights_blockwise_multi_host,
    selftest_bounded_wait,
    silu_mul_bf16,
    silu_mul_quantize,
    tis_weights,
    version,
    weight_shard_rows,
)
from . import weight_sync  # noqa: F401
