"""Seeded synthetic inputs for the FP8 rollout hot path.

This module only draws random numbers with torch's generators and arranges
them into the shapes of the workloads; it holds none of the quantization,
GEMM or importance-weight arithmetic, so both the CUDA path and the CPU
oracle may consume what it produces.

Workloads (synthetic stand-ins for the models the FP8-RL pages train:
Qwen3-8B-Base and Qwen3-30B-A3B-Base; no weights or datasets are used):

* ``tiny_linear``   -- A bf16 [64, 512] ~ N(0,1) with 1% of columns x20,
  W bf16 [256, 512] ~ N(0, 0.02); TIS on 4096 tokens.
* ``qwen3_8b_linear_shapes`` / ``make_weight`` -- the four quantized linear
  shapes of one Qwen3-8B layer (36 layers), bf16 ~ N(0, 0.02) with 0.1% of
  entries x50.
* ``dense_acts``    -- activations bf16 ~ N(0,1) times a per-token
  LogNormal(0,1) factor.
* ``moe_routing`` / ``moe_weights`` -- Qwen3-30B-A3B expert FFN shapes, 128
  experts, 4096 tokens routed top-8 by router logits N(0,1) plus a Zipf(1.1)
  per-expert bias (skewed expert loads).
* ``kv_tensor``     -- one layer's K or V [S, T, 8, 128] bf16 ~ N(0,1) with 5%
  of (head, dim) channels x10.
* ``tis_logprobs``  -- rollout log-probs -|N(0,2)|, training log-probs shifted
  by N(0, 0.05) or by 0.05 * Student-t(3).
"""
from __future__ import annotations

import math

import torch

QWEN3_8B_LAYERS = 36
QWEN3_8B_HIDDEN = 4096
# (name, N, K) of the quantized linears of one Qwen3-8B layer: fused q/k/v,
# o_proj, fused gate/up, down_proj (nn.Linear weight layout [out, in]).
QWEN3_8B_LINEARS = (
    ("qkv", 6144, 4096),
    ("o", 4096, 4096),
    ("gate_up", 24576, 4096),
    ("down", 4096, 12288),
)

MOE_EXPERTS = 128
MOE_HIDDEN = 2048
MOE_INTER = 768
MOE_TOKENS = 4096
MOE_TOPK = 8


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def sub_seed(*parts: int) -> int:
    """Deterministic sub-seed from integer parts (layer, tensor, ...)."""
    h = 1469598103934665603
    for p in parts:
        h = ((h ^ (int(p) & 0xFFFFFFFFFFFF)) * 1099511628211) % (1 << 63)
    return h


def tiny_linear(seed: int = 0, device="cpu", m: int = 64, n: int = 256, k: int = 512):
    """A [m, k] ~ N(0,1) with 1% of columns x20 (outlier channels); W [n, k] ~ N(0, 0.02)."""
    g = _gen(seed, device)
    a = torch.randn(m, k, generator=g, device=device)
    n_out = max(1, round(0.01 * k))
    cols = torch.randperm(k, generator=g, device=device)[:n_out]
    a[:, cols] *= 20.0
    w = torch.randn(n, k, generator=g, device=device) * 0.02
    return a.to(torch.bfloat16), w.to(torch.bfloat16)


def qwen3_8b_linear_shapes(layers: int = QWEN3_8B_LAYERS):
    """[(layer, name, N, K)] for every quantized linear of Qwen3-8B."""
    return [(l, name, n, k) for l in range(layers) for (name, n, k) in QWEN3_8B_LINEARS]


def make_weight(n: int, k: int, seed: int, device="cpu", std: float = 0.02,
                outlier_frac: float = 0.001, outlier_mult: float = 50.0):
    """bf16 [n, k] ~ N(0, std) with a random outlier_frac of entries multiplied."""
    g = _gen(seed, device)
    w = torch.randn(n, k, generator=g, device=device)
    w.mul_(std)
    if outlier_frac > 0:
        mask = torch.rand(n, k, generator=g, device=device) < outlier_frac
        w = torch.where(mask, w * outlier_mult, w)
    return w.to(torch.bfloat16)


def dense_acts(m: int, k: int, seed: int, device="cpu"):
    """bf16 [m, k]: N(0,1) entries times a per-token LogNormal(0,1) factor."""
    g = _gen(seed, device)
    a = torch.randn(m, k, generator=g, device=device)
    tok = torch.exp(torch.randn(m, 1, generator=g, device=device))
    return (a * tok).to(torch.bfloat16)


def moe_routing(seed: int = 0, tokens: int = MOE_TOKENS, experts: int = MOE_EXPERTS,
                topk: int = MOE_TOPK, zipf_s: float = 1.1):
    """Top-k routing with Zipf-skewed expert popularity.

    Router logits are N(0,1) plus a per-expert bias -zipf_s * ln(rank), the rank a
    seeded permutation of 1..experts, so that softmax preference falls off like
    rank^-zipf_s.  Top-k by logit (softmax is monotone); rows are packed by
    expert, then by (token, slot).  Returns (offsets int32 [experts+1],
    token_of_row int64 [tokens*topk], counts int64 [experts]).
    """
    g = _gen(seed, "cpu")
    logits = torch.randn(tokens, experts, generator=g, dtype=torch.float64)
    rank = torch.randperm(experts, generator=g).to(torch.float64) + 1.0
    logits = logits - zipf_s * torch.log(rank)[None, :]
    top = torch.topk(logits, topk, dim=1).indices            # [tokens, topk]
    expert_of = top.reshape(-1)
    token_of = torch.arange(tokens).repeat_interleave(topk)
    order = torch.argsort(expert_of * (tokens * topk) + torch.arange(tokens * topk), stable=True)
    counts = torch.bincount(expert_of, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    return offsets.to(torch.int32), token_of[order], counts


def moe_weights(n: int, k: int, experts: int, seed: int, device="cpu", std: float = 0.02):
    """bf16 [experts, n, k] ~ N(0, std)."""
    g = _gen(seed, device)
    w = torch.randn(experts, n, k, generator=g, device=device)
    w.mul_(std)
    return w.to(torch.bfloat16)


def expert_inputs(rows: int, k: int, seed: int, device="cpu"):
    """Packed expert inputs bf16 [rows, k] ~ N(0,1)."""
    g = _gen(seed, device)
    return torch.randn(rows, k, generator=g, device=device).to(torch.bfloat16)


def kv_tensor(seed: int, device="cpu", seqs: int = 64, tokens: int = 20480, heads: int = 8,
              head_dim: int = 128, outlier_frac: float = 0.05, outlier_mult: float = 10.0):
    """bf16 [seqs, tokens, heads, head_dim] ~ N(0,1); a fixed 5% of the
    (head, dim) channels are multiplied for every token (outlier channels)."""
    g = _gen(seed, device)
    ch = heads * head_dim
    n_out = int(math.floor(outlier_frac * ch))
    sel = torch.randperm(ch, generator=g, device=device)[:n_out]
    mult = torch.ones(ch, device=device)
    mult[sel] = outlier_mult
    x = torch.empty(seqs, tokens, heads, head_dim, dtype=torch.bfloat16, device=device)
    step = max(1, (1 << 26) // (tokens * ch))        # generate a few sequences at a time
    for s0 in range(0, seqs, step):
        s1 = min(seqs, s0 + step)
        blk = torch.randn(s1 - s0, tokens, ch, generator=g, device=device)
        blk.mul_(mult)
        x[s0:s1] = blk.view(s1 - s0, tokens, heads, head_dim).to(torch.bfloat16)
    return x


def tis_logprobs(n: int, seed: int, device="cpu", kind: str = "normal"):
    """(logp_train, logp_rollout) float32 [n].

    logp_rollout = -|N(0, 2)|.  kind="normal": logp_train = logp_rollout +
    N(0, 0.05); kind="student_t": the shift is 0.05 * t with nu = 3, drawn as
    Z / sqrt(chi2_3 / 3).
    """
    g = _gen(seed, device)
    lr = -torch.abs(torch.randn(n, generator=g, device=device) * 2.0)
    if kind == "normal":
        d = torch.randn(n, generator=g, device=device) * 0.05
    elif kind == "student_t":
        z = torch.randn(n, generator=g, device=device)
        c = (torch.randn(3, n, generator=g, device=device) ** 2).sum(0) / 3.0
        d = 0.05 * z / torch.sqrt(c)
    else:
        raise ValueError(kind)
    lt = lr + d
    return lt.to(torch.float32), lr.to(torch.float32)
