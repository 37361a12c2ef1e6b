"""Thin ctypes binding of libfp8rl.so with the C ABI's call names.

Argument marshalling only: every function checks dtypes/devices of the torch
tensors it is given, allocates missing outputs with torch (device memory is
torch's job here), and passes raw pointers plus the current CUDA stream to the
library.  Every step of the computation runs in the library's kernels.  If the
library is missing or fails to load, the first call raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8rl.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "fp8rl.h")

FP8RL_OK = 0
FP8RL_KV_GIVEN = 0
FP8RL_KV_CALIBRATE = 1
FP8RL_IS_TRUNCATE = 0
FP8RL_IS_MASK = 1
_STATUS = {0: "FP8RL_OK", 1: "FP8RL_ERR_INVALID_ARG", 2: "FP8RL_ERR_ALIGNMENT",
           3: "FP8RL_ERR_UNSUPPORTED_SHAPE", 4: "FP8RL_ERR_CUDA", 5: "FP8RL_ERR_TIMEOUT",
           6: "FP8RL_ERR_UNSUPPORTED_DEVICE"}


class Fp8rlError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, str(status)), message))
        self.status = status


class WDesc(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("q", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("ldq", ctypes.c_int64)]


_lib = None


def load(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of libfp8rl.so."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libfp8rl.so not found at %s: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % p)
    L = ctypes.CDLL(p)
    P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    sigs = {
        "fp8rl_version": (i32, []),
        "fp8rl_last_error": (ctypes.c_char_p, []),
        "fp8rl_quantize_weights_blockwise": (ctypes.c_int, [P, i64, i64, i64, P, i64, P, P]),
        "fp8rl_quantize_weights_blockwise_multi": (ctypes.c_int, [P, i32, P]),
        "fp8rl_quantize_act_groupwise": (ctypes.c_int, [P, i64, i64, i64, P, P, P]),
        "fp8rl_gemm_w8a8_blockwise": (ctypes.c_int, [P, P, P, P, i64, i64, i64, P, i64, P]),
        "fp8rl_grouped_gemm_w8a8_blockwise": (ctypes.c_int, [P, P, P, P, P, i32, i64, i64, i64,
                                                              P, P]),
        "fp8rl_quantize_kv_fp8": (ctypes.c_int, [P, i64, i32, i32, i32, P, P, P]),
        "fp8rl_tis_weights": (ctypes.c_int, [P, P, P, i64, f32, f32, P, P]),
        "fp8rl_is_weights_stats": (ctypes.c_int, [P, P, P, i64, f32, f32, i32, P, P, P]),
        "fp8rl_is_weights_stats_loss": (ctypes.c_int, [P, P, P, P, i64, f32, f32, i32, P, P, P]),
        "fp8rl_quantize_act_gather": (ctypes.c_int, [P, i64, i64, i64, P, i64, P, P, P]),
        "fp8rl_quantize_weights_blockwise_multi_host": (ctypes.c_int, [P, i32, P, ctypes.c_size_t,
                                                                       P]),
        "fp8rl_silu_mul_quantize": (ctypes.c_int, [P, i64, i64, i64, P, P, P]),
        "fp8rl_silu_mul_bf16": (ctypes.c_int, [P, i64, i64, i64, P, i64, P]),
        "fp8rl_linear_w8a8_decode_workspace_bytes": (ctypes.c_size_t, [i64]),
        "fp8rl_linear_w8a8_decode": (ctypes.c_int, [P, i64, P, P, P, P, i64, i64, i64, P, i64, P,
                                                    ctypes.c_size_t, P]),
        "fp8rl_decode_attention_fp8kv": (ctypes.c_int, [P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                        i32, i32, i32, f32, P, P]),
        "fp8rl_device_status": (ctypes.c_int, [i32, i32]),
        "fp8rl_weight_shard_rows": (ctypes.c_int, [i64, i32, i32, P, P]),
        "fp8rl_inject_device_status": (ctypes.c_int, [i32, ctypes.c_uint32, ctypes.c_uint32]),
        "fp8rl_selftest_bounded_wait": (ctypes.c_int, [i32, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = L
    return L


def declared_symbols(header: str = HEADER) -> list:
    """Names of the functions include/fp8rl.h declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"\b(fp8rl_[a-z0-9_]+)\s*\(", text)))


def last_error() -> str:
    return load().fp8rl_last_error().decode()


def version() -> int:
    return int(load().fp8rl_version())


def _check(status: int):
    if status != FP8RL_OK:
        raise Fp8rlError(status, last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _rowmajor(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a 2-D tensor with unit column stride" % name)
    return t


# -------------------------------------------------------------- quantizers --

def quantize_weights_blockwise(w: torch.Tensor, q: Optional[torch.Tensor] = None,
                               scales: Optional[torch.Tensor] = None, stream=None):
    """128x128-block E4M3 quantization of a bf16 [n, k] weight -> (codes uint8, scales f32)."""
    _rowmajor(_dev(w, torch.bfloat16, "w"), "w")
    n, k = w.shape
    if q is None:
        q = torch.empty(n, k, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((n + 127) // 128, (k + 127) // 128, dtype=torch.float32, device=w.device)
    _rowmajor(_dev(q, torch.uint8, "q"), "q")
    _dev(scales, torch.float32, "scales")
    _check(load().fp8rl_quantize_weights_blockwise(w.data_ptr(), n, k, w.stride(0), q.data_ptr(),
                                                   q.stride(0), scales.data_ptr(), _stream(stream)))
    return q, scales


def quantize_weights_blockwise_multi(ws: Sequence[torch.Tensor], qs=None, ss=None, stream=None):
    """One launch over many weights (a whole model's per-step re-quantization)."""
    ws = list(ws)
    qs = list(qs) if qs is not None else [torch.empty(w.shape, dtype=torch.uint8, device=w.device)
                                          for w in ws]
    ss = list(ss) if ss is not None else [
        torch.empty((w.shape[0] + 127) // 128, (w.shape[1] + 127) // 128, dtype=torch.float32,
                    device=w.device) for w in ws]
    arr = (WDesc * max(1, len(ws)))()
    for i, (w, q, s) in enumerate(zip(ws, qs, ss)):
        _rowmajor(_dev(w, torch.bfloat16, "w[%d]" % i), "w")
        _rowmajor(_dev(q, torch.uint8, "q[%d]" % i), "q")
        _dev(s, torch.float32, "scales[%d]" % i)
        arr[i] = WDesc(w.data_ptr(), q.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1],
                       w.stride(0), q.stride(0))
    _check(load().fp8rl_quantize_weights_blockwise_multi(ctypes.addressof(arr), len(ws),
                                                         _stream(stream)))
    return qs, ss


def quantize_act_groupwise(a: torch.Tensor, q: Optional[torch.Tensor] = None,
                           scales: Optional[torch.Tensor] = None, stream=None):
    """Per-token 1x128 E4M3 quantization of bf16 [m, k] -> (codes [m, k], scales [ceil(k/128), m])."""
    _rowmajor(_dev(a, torch.bfloat16, "a"), "a")
    m, k = a.shape
    if q is None:
        q = torch.empty(m, k, dtype=torch.uint8, device=a.device)
    if scales is None:
        scales = torch.empty((k + 127) // 128, m, dtype=torch.float32, device=a.device)
    _dev(q, torch.uint8, "q")
    _dev(scales, torch.float32, "scales")
    if not q.is_contiguous():
        raise ValueError("q must be dense [m, k]")
    _check(load().fp8rl_quantize_act_groupwise(a.data_ptr(), m, k, a.stride(0), q.data_ptr(),
                                               scales.data_ptr(), _stream(stream)))
    return q, scales


def quantize_kv_fp8(x: torch.Tensor, mode: int = FP8RL_KV_CALIBRATE,
                    scales: Optional[torch.Tensor] = None, q: Optional[torch.Tensor] = None,
                    stream=None):
    """E4M3 K or V cache of bf16 [..., heads, head_dim] with per-head scales -> (codes, scales)."""
    _dev(x, torch.bfloat16, "x")
    if not x.is_contiguous() or x.dim() < 2:
        raise ValueError("x must be a dense [..., heads, head_dim] tensor")
    heads, hd = x.shape[-2], x.shape[-1]
    rows = x.numel() // (heads * hd)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        if mode == FP8RL_KV_GIVEN:
            raise ValueError("FP8RL_KV_GIVEN needs scales")
        scales = torch.empty(heads, dtype=torch.float32, device=x.device)
    _dev(q, torch.uint8, "q")
    _dev(scales, torch.float32, "scales")
    _check(load().fp8rl_quantize_kv_fp8(x.data_ptr(), rows, heads, hd, mode, scales.data_ptr(),
                                        q.data_ptr(), _stream(stream)))
    return q, scales


# ------------------------------------------------------------------ GEMMs --

def gemm_w8a8_blockwise(qa, sa, qw, sw, y: Optional[torch.Tensor] = None, stream=None):
    """Y = A W^T (bf16 [m, n]) from E4M3 codes and their block scales."""
    _dev(qa, torch.uint8, "qa"); _dev(qw, torch.uint8, "qw")
    _dev(sa, torch.float32, "sa"); _dev(sw, torch.float32, "sw")
    m, k = qa.shape
    n = qw.shape[0]
    if y is None:
        y = torch.empty(m, n, dtype=torch.bfloat16, device=qa.device)
    _rowmajor(_dev(y, torch.bfloat16, "y"), "y")
    _check(load().fp8rl_gemm_w8a8_blockwise(qa.data_ptr(), sa.data_ptr(), qw.data_ptr(),
                                            sw.data_ptr(), m, n, k, y.data_ptr(), y.stride(0),
                                            _stream(stream)))
    return y


def linear_w8a8_decode_workspace_bytes(n: int) -> int:
    """Workspace bytes linear_w8a8_decode needs for n output columns on the
    current device."""
    return int(load().fp8rl_linear_w8a8_decode_workspace_bytes(int(n)))


def linear_w8a8_decode(a, qw, sw, y: Optional[torch.Tensor] = None,
                       qa: Optional[torch.Tensor] = None, sa: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None):
    """Decode-sized linear layer (m <= 256): quantize bf16 a [m, k] in 1x128
    groups and multiply by the E4M3 weights in one launch.  Returns (y, qa, sa).
    With a=None, qa/sa are the (already quantized) inputs.  workspace: a
    zero-filled uint8 device tensor of linear_w8a8_decode_workspace_bytes(n)
    bytes, reusable across calls (allocated here when None)."""
    _dev(qw, torch.uint8, "qw"); _dev(sw, torch.float32, "sw")
    n, k = qw.shape
    dev = qw.device
    if a is not None:
        _rowmajor(_dev(a, torch.bfloat16, "a"), "a")
        m = a.shape[0]
        if qa is None:
            qa = torch.empty(m, k, dtype=torch.uint8, device=dev)
        if sa is None:
            sa = torch.empty(k // 128, m, dtype=torch.float32, device=dev)
    else:
        if qa is None or sa is None:
            raise ValueError("without a, qa and sa are required")
        m = qa.shape[0]
    _dev(qa, torch.uint8, "qa"); _dev(sa, torch.float32, "sa")
    if y is None:
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    _rowmajor(_dev(y, torch.bfloat16, "y"), "y")
    if workspace is None:
        workspace = torch.zeros(linear_w8a8_decode_workspace_bytes(n), dtype=torch.uint8, device=dev)
    _dev(workspace, torch.uint8, "workspace")
    _check(load().fp8rl_linear_w8a8_decode(a.data_ptr() if a is not None else None,
                                           a.stride(0) if a is not None else k,
                                           qa.data_ptr(), sa.data_ptr(), qw.data_ptr(),
                                           sw.data_ptr(), m, n, k, y.data_ptr(), y.stride(0),
                                           workspace.data_ptr(), workspace.numel(),
                                           _stream(stream)))
    return y, qa, sa


def grouped_gemm_w8a8_blockwise(qa, sa, qw, sw, offsets, y: Optional[torch.Tensor] = None,
                                stream=None):
    """Per-expert Y rows: rows [offsets[e], offsets[e+1]) use expert e's weights."""
    _dev(qa, torch.uint8, "qa"); _dev(qw, torch.uint8, "qw")
    _dev(sa, torch.float32, "sa"); _dev(sw, torch.float32, "sw")
    _dev(offsets, torch.int32, "offsets")
    m, k = qa.shape
    e, n, _ = qw.shape
    if y is None:
        y = torch.empty(m, n, dtype=torch.bfloat16, device=qa.device)
    _dev(y, torch.bfloat16, "y")
    _check(load().fp8rl_grouped_gemm_w8a8_blockwise(qa.data_ptr(), sa.data_ptr(), qw.data_ptr(),
                                                    sw.data_ptr(), offsets.data_ptr(), e, m, n,
                                                    k, y.data_ptr(), _stream(stream)))
    return y


def quantize_weights_blockwise_multi_host(ws, qs, ss, workspace: torch.Tensor, stream=None):
    """Re-quantize HOST BF16 weights ws[i] [n, k] into HOST codes qs[i] and
    scales ss[i], streaming through the device `workspace` (uint8 tensor);
    copies and kernels overlap.  Host tensors should be pinned."""
    if not (len(ws) == len(qs) == len(ss)):
        raise ValueError("ws, qs and ss must have the same length")
    _dev(workspace, torch.uint8, "workspace")
    arr = (WDesc * max(len(ws), 1))()
    for i, (w, q, s) in enumerate(zip(ws, qs, ss)):
        for t, name, dt in ((w, "w", torch.bfloat16), (q, "q", torch.uint8), (s, "scales", torch.float32)):
            if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dt:
                raise TypeError("%s[%d] must be a host %s tensor" % (name, i, dt))
        _rowmajor(w, "w"); _rowmajor(q, "q")
        if not s.is_contiguous():
            raise ValueError("scales must be contiguous")
        n, k = w.shape
        arr[i] = WDesc(w.data_ptr(), q.data_ptr(), s.data_ptr(), n, k, w.stride(0), q.stride(0))
    _check(load().fp8rl_quantize_weights_blockwise_multi_host(
        ctypes.cast(arr, ctypes.c_void_p), len(ws), workspace.data_ptr(), workspace.numel(),
        _stream(stream)))


# --------------------------------------------------------------- MoE glue --

def quantize_act_gather(a, rows, q: Optional[torch.Tensor] = None,
                        scales: Optional[torch.Tensor] = None, stream=None):
    """Codes and group-major scales of the gathered rows a[rows[r]] (1x128 groups)."""
    _dev(a, torch.bfloat16, "a")
    _rowmajor(a, "a")
    _dev(rows, torch.int32, "rows")
    if not rows.is_contiguous():
        raise ValueError("rows must be contiguous")
    m_src, k = a.shape
    m = rows.numel()
    if q is None:
        q = torch.empty(m, k, dtype=torch.uint8, device=a.device)
    if scales is None:
        scales = torch.empty((k + 127) // 128, m, dtype=torch.float32, device=a.device)
    _dev(q, torch.uint8, "q"); _dev(scales, torch.float32, "scales")
    _check(load().fp8rl_quantize_act_gather(a.data_ptr(), m_src, k, a.stride(0), rows.data_ptr(),
                                            m, q.data_ptr(), scales.data_ptr(), _stream(stream)))
    return q, scales


def silu_mul_quantize(h, q: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                      stream=None):
    """h = [gate | up] BF16 [m, 2*inter] -> codes and group-major scales of
    BF16(silu(gate) * up)."""
    _dev(h, torch.bfloat16, "h")
    _rowmajor(h, "h")
    m, two_i = h.shape
    if two_i % 2:
        raise ValueError("h must have an even number of columns (gate | up)")
    inter = two_i // 2
    if q is None:
        q = torch.empty(m, inter, dtype=torch.uint8, device=h.device)
    if scales is None:
        scales = torch.empty((inter + 127) // 128, m, dtype=torch.float32, device=h.device)
    _dev(q, torch.uint8, "q"); _dev(scales, torch.float32, "scales")
    _check(load().fp8rl_silu_mul_quantize(h.data_ptr(), m, inter, h.stride(0), q.data_ptr(),
                                          scales.data_ptr(), _stream(stream)))
    return q, scales


def silu_mul_bf16(h, y: Optional[torch.Tensor] = None, stream=None):
    """h = [gate | up] BF16 [m, 2*inter] -> y = BF16_RNE(silu(gate) * up), BF16 [m, inter]."""
    _dev(h, torch.bfloat16, "h")
    _rowmajor(h, "h")
    m, two_i = h.shape
    if two_i % 2:
        raise ValueError("h must have an even number of columns (gate | up)")
    inter = two_i // 2
    if y is None:
        y = torch.empty(m, inter, dtype=torch.bfloat16, device=h.device)
    _rowmajor(_dev(y, torch.bfloat16, "y"), "y")
    _check(load().fp8rl_silu_mul_bf16(h.data_ptr(), m, inter, h.stride(0), y.data_ptr(),
                                      y.stride(0), _stream(stream)))
    return y


# -------------------------------------------------------------- attention --

def decode_attention_fp8kv(q, k_cache, v_cache, k_scale, v_scale, seq_lens, block_table=None,
                           sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                           stream=None):
    """Decode attention of q BF16 [S, Hq, 128] over an E4M3 cache
    [pages, page, Hkv, 128] (k_cache, v_cache, per-head scales [Hkv]).
    block_table int32 [S, max_pages] or None (contiguous: the cache is
    [S, T, Hkv, 128], or [S*T, Hkv, 128] rows as the KV quantizer writes)."""
    _dev(q, torch.bfloat16, "q")
    _dev(k_cache, torch.uint8, "k_cache"); _dev(v_cache, torch.uint8, "v_cache")
    _dev(k_scale, torch.float32, "k_scale"); _dev(v_scale, torch.float32, "v_scale")
    _dev(seq_lens, torch.int32, "seq_lens")
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("q and the caches must be contiguous")
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
        raise ValueError("caches must be [pages, page, kv_heads, head_dim] and equal in shape")
    S, hq, d = q.shape
    pages, page, hkv, _ = k_cache.shape
    if block_table is None:
        if pages != S:
            raise ValueError("a contiguous cache needs one page per sequence")
        tp, max_pages = 0, 1
    else:
        _dev(block_table, torch.int32, "block_table")
        if block_table.dim() != 2 or block_table.shape[0] != S or not block_table.is_contiguous():
            raise ValueError("block_table must be a contiguous [S, max_pages] tensor")
        tp, max_pages = block_table.data_ptr(), block_table.shape[1]
    if out is None:
        out = torch.empty(S, hq, d, dtype=torch.bfloat16, device=q.device)
    _dev(out, torch.bfloat16, "out")
    if sm_scale is None:
        sm_scale = d ** -0.5
    _check(load().fp8rl_decode_attention_fp8kv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                               k_scale.data_ptr(), v_scale.data_ptr(), tp,
                                               seq_lens.data_ptr(), S, hq, hkv, d, page, max_pages,
                                               pages, float(sm_scale), out.data_ptr(),
                                               _stream(stream)))
    return out


# --------------------------------------------------------------------- TIS --

def tis_weights(logp_train, logp_rollout, mask=None, c_hi: float = 2.0, c_lo: float = 0.0,
                w: Optional[torch.Tensor] = None, stream=None):
    """Truncated importance weights min(exp(lt - lr), c_hi) (and >= c_lo when c_lo > 0)."""
    _dev(logp_train, torch.float32, "logp_train")
    _dev(logp_rollout, torch.float32, "logp_rollout")
    n = logp_train.numel()
    if logp_rollout.numel() != n:
        raise ValueError("logp_train and logp_rollout must have the same size")
    if w is None:
        w = torch.empty_like(logp_train)
    _dev(w, torch.float32, "w")
    mp = 0
    if mask is not None:
        _dev(mask, torch.uint8, "mask")
        mp = mask.data_ptr()
    _check(load().fp8rl_tis_weights(logp_train.data_ptr(), logp_rollout.data_ptr(), mp, n,
                                    float(c_hi), float(c_lo), w.data_ptr(), _stream(stream)))
    return w


def is_weights_stats(logp_train, logp_rollout, mask=None, c_hi: float = 2.0, c_lo: float = 0.0,
                     mode: int = FP8RL_IS_TRUNCATE, w: Optional[torch.Tensor] = None,
                     stats: Optional[torch.Tensor] = None, weights: bool = True, stream=None,
                     loss: Optional[torch.Tensor] = None):
    """Importance weights (TIS or MIS by `mode`) and the batch's mismatch
    statistics [valid tokens, sum k1, sum k3, sum of ratios, clipped/masked
    tokens] (float64 [5]); with a per-token `loss` (float32 [n]) a sixth entry,
    the sum of fl32(w * loss) over the valid tokens.  weights=False computes
    the statistics only.  Returns (w or None, stats)."""
    _dev(logp_train, torch.float32, "logp_train")
    _dev(logp_rollout, torch.float32, "logp_rollout")
    n = logp_train.numel()
    if logp_rollout.numel() != n:
        raise ValueError("logp_train and logp_rollout must have the same size")
    wp = 0
    if weights:
        if w is None:
            w = torch.empty_like(logp_train)
        _dev(w, torch.float32, "w")
        wp = w.data_ptr()
    else:
        w = None
    nstats = 5 if loss is None else 6
    if stats is None:
        stats = torch.empty(nstats, dtype=torch.float64, device=logp_train.device)
    _dev(stats, torch.float64, "stats")
    if stats.numel() < nstats:
        raise ValueError("stats must hold %d values" % nstats)
    mp = 0
    if mask is not None:
        _dev(mask, torch.uint8, "mask")
        mp = mask.data_ptr()
    if loss is None:
        _check(load().fp8rl_is_weights_stats(logp_train.data_ptr(), logp_rollout.data_ptr(), mp, n,
                                             float(c_hi), float(c_lo), int(mode), wp,
                                             stats.data_ptr(), _stream(stream)))
    else:
        _dev(loss, torch.float32, "loss")
        if loss.numel() != n:
            raise ValueError("loss must have one value per token")
        _check(load().fp8rl_is_weights_stats_loss(logp_train.data_ptr(), logp_rollout.data_ptr(),
                                                  mp, loss.data_ptr(), n, float(c_hi),
                                                  float(c_lo), int(mode), wp, stats.data_ptr(),
                                                  _stream(stream)))
    return w, stats


def is_weights_stats_loss(logp_train, logp_rollout, loss, mask=None, c_hi: float = 2.0,
                          c_lo: float = 0.0, mode: int = FP8RL_IS_TRUNCATE,
                          w: Optional[torch.Tensor] = None, stats: Optional[torch.Tensor] = None,
                          weights: bool = True, stream=None):
    """is_weights_stats with the importance-weighted token loss as a sixth
    statistic (sum of fl32(w * loss) over the valid tokens)."""
    return is_weights_stats(logp_train, logp_rollout, mask, c_hi, c_lo, mode, w, stats, weights,
                            stream, loss=loss)


def quantize_kv_fp8_calibrate_noalloc(x: torch.Tensor, scales: Optional[torch.Tensor] = None,
                                      q: Optional[torch.Tensor] = None, stream=None):
    """KV calibrate + quantize without any device allocation by the library
    (scratch is a fixed 256-head array inside it); same results as
    quantize_kv_fp8(x, FP8RL_KV_CALIBRATE)."""
    _dev(x, torch.bfloat16, "x")
    if not x.is_contiguous() or x.dim() < 2:
        raise ValueError("x must be a dense [..., heads, head_dim] tensor")
    heads, hd = x.shape[-2], x.shape[-1]
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(heads, dtype=torch.float32, device=x.device)
    fn = load().fp8rl_quantize_kv_fp8_calibrate_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    _check(fn(x.data_ptr(), x.numel() // (heads * hd), heads, hd, scales.data_ptr(), q.data_ptr(),
              _stream(stream)))
    return q, scales


def device_status(device: int = 0, clear: bool = True) -> int:
    """Raises Fp8rlError(FP8RL_ERR_TIMEOUT) if a kernel hit a device-side wait limit."""
    st = load().fp8rl_device_status(device, 1 if clear else 0)
    _check(st)
    return st


def inject_device_status(device: int, flags: int, site: int = 0):
    """Overwrite the device status word (error-path tests; see fp8rl.h)."""
    _check(load().fp8rl_inject_device_status(device, flags, site))


def selftest_bounded_wait(limit_us: int, stream=None):
    """Launch the bounded-wait self-test kernel (its wait times out; see fp8rl.h)."""
    _check(load().fp8rl_selftest_bounded_wait(int(limit_us), _stream(stream)))


def weight_shard_rows(n: int, world: int, rank: int):
    """Rows [begin, end) of an n-row weight owned by `rank` in the sharded
    weight sync (whole 128-row block bands; see fp8rl.h)."""
    b, e = ctypes.c_int64(), ctypes.c_int64()
    _check(load().fp8rl_weight_shard_rows(int(n), int(world), int(rank), ctypes.byref(b),
                                          ctypes.byref(e)))
    return b.value, e.value
