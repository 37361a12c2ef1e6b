"""GB300-native hot path of the FP8 RL rollout stack (FP8-RL, arXiv 2601.18150).

The compute lives in a C-ABI CUDA library (``libfp8rl.so``, sources in
``csrc/``, declarations in ``include/fp8rl.h``); :mod:`.binding` is a thin
ctypes layer with the same call names.  The library is loaded on the first
call and a missing or unloadable library raises -- there is no fallback.
"""
__all__ = ["workloads"]
