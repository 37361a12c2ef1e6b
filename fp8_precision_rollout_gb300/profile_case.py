"""Run one hot-path kernel on a fixed small-but-larger-than-L2 case, for
profiler captures (ncu) of a single kernel.  Prints nothing but a done line;
timing numbers come from bench.py, never from here.

    python -m fp8_precision_rollout_gb300.profile_case CASE [--iters N]

Cases (device footprint in parentheses):
  wquant          re-quantization of Qwen3-8B layer-0 linears, one launch (0.6 GB)
  aquant          1x128 activation quantization, M=8192 K=4096 (0.1 GB)
  gemm_prefill    act-quant'ed W8A8 GEMM, gate_up shape M=8192 N=24576 K=4096 (0.6 GB)
  gemm_decode     W8A8 GEMM, qkv shape M=256 N=6144 K=4096 (0.03 GB)
  gemm_decode_o   W8A8 GEMM, o shape M=256 N=4096 K=4096 (0.02 GB; split-K clusters of 2)
  linear_decode   fused act-quant + stream-K W8A8 GEMM, qkv shape M=256 N=6144 K=4096 (0.03 GB)
  linear_decode_o the same, o shape M=256 N=4096 K=4096 (0.02 GB)
  grouped         grouped W8A8 GEMM, Qwen3-30B-A3B gate_up, 128 experts (0.5 GB)
  kv              KV calibrate + quantize, 8 x 20480 tokens x 8 x 128 (0.5 GB)
  tis             TIS weights over 64 x 20480 tokens (0.02 GB)
  is_stats        MIS weights + mismatch statistics + weighted token loss, 64 x 20480 tokens
                  (0.02 GB)
  attention       FP8-KV decode attention, 64 seqs x 4096 tokens, 32 q / 8 KV heads (0.6 GB;
                  one CTA per sequence and KV head, as at 64 x 20480)
  glue_gather     MoE gather + quantize: 4096 tokens x 2048 -> 32768 routed rows (0.1 GB)
  glue_silu       MoE SiLU(gate)*up + quantize: 32768 x 1536 -> 32768 x 768 (0.13 GB)
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402

import fp8_precision_rollout_gb300 as fp8rl  # noqa: E402
from fp8_precision_rollout_gb300 import workloads as wl  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    c = args.case
    if c == "wquant":
        ws = [wl.make_weight(n, k, seed=wl.sub_seed(2, 0, i), device=dev)
              for i, (_, n, k) in enumerate(wl.QWEN3_8B_LINEARS)]
        qs = [torch.empty(w.shape, dtype=torch.uint8, device=dev) for w in ws]
        ss = [torch.empty(w.shape[0] // 128, w.shape[1] // 128, dtype=torch.float32, device=dev)
              for w in ws]
        run = lambda: fp8rl.quantize_weights_blockwise_multi(ws, qs, ss)  # noqa: E731
    elif c == "aquant":
        a = wl.dense_acts(8192, 4096, seed=1, device=dev)
        run = lambda: fp8rl.quantize_act_groupwise(a)  # noqa: E731
    elif c in ("gemm_prefill", "gemm_decode", "gemm_decode_o"):
        m, n, k = {"gemm_prefill": (8192, 24576, 4096), "gemm_decode": (256, 6144, 4096),
                   "gemm_decode_o": (256, 4096, 4096)}[c]
        qa, sa = fp8rl.quantize_act_groupwise(wl.dense_acts(m, k, seed=2, device=dev))
        qw, sw = fp8rl.quantize_weights_blockwise(wl.make_weight(n, k, seed=3, device=dev))
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        run = lambda: fp8rl.gemm_w8a8_blockwise(qa, sa, qw, sw, y)  # noqa: E731
    elif c in ("linear_decode", "linear_decode_o"):
        m, n, k = (256, 6144, 4096) if c == "linear_decode" else (256, 4096, 4096)
        a = wl.dense_acts(m, k, seed=2, device=dev)
        qw, sw = fp8rl.quantize_weights_blockwise(wl.make_weight(n, k, seed=3, device=dev))
        y = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        qa = torch.empty(m, k, dtype=torch.uint8, device=dev)
        sa = torch.empty(k // 128, m, dtype=torch.float32, device=dev)
        ws = torch.zeros(fp8rl.linear_w8a8_decode_workspace_bytes(n), dtype=torch.uint8, device=dev)
        run = lambda: fp8rl.linear_w8a8_decode(a, qw, sw, y, qa, sa, ws)  # noqa: E731
    elif c == "grouped":
        off, _, _ = wl.moe_routing(seed=0)
        rows = int(off[-1])
        n, k, e = 2 * wl.MOE_INTER, wl.MOE_HIDDEN, wl.MOE_EXPERTS
        qa, sa = fp8rl.quantize_act_groupwise(wl.expert_inputs(rows, k, seed=4, device=dev))
        qw, sw = fp8rl.quantize_weights_blockwise(wl.moe_weights(n, k, e, seed=5, device=dev)
                                                  .view(-1, k))
        offd = off.to(dev)
        y = torch.empty(rows, n, dtype=torch.bfloat16, device=dev)
        run = lambda: fp8rl.grouped_gemm_w8a8_blockwise(  # noqa: E731
            qa, sa, qw.view(e, n, k), sw.view(e, n // 128, k // 128), offd, y)
    elif c == "kv":
        x = wl.kv_tensor(seed=6, device=dev, seqs=8)
        run = lambda: fp8rl.quantize_kv_fp8(x, fp8rl.FP8RL_KV_CALIBRATE)  # noqa: E731
    elif c == "tis":
        lt, lr = wl.tis_logprobs(64 * 20480, seed=5, device=dev, kind="student_t")
        run = lambda: fp8rl.tis_weights(lt, lr)  # noqa: E731
    elif c == "is_stats":
        lt, lr = wl.tis_logprobs(64 * 20480, seed=5, device=dev, kind="student_t")
        loss = torch.randn(lt.numel(), generator=torch.Generator().manual_seed(8)).to(dev)
        w = torch.empty(lt.numel(), dtype=torch.float32, device=dev)
        stats = torch.empty(6, dtype=torch.float64, device=dev)
        run = lambda: fp8rl.is_weights_stats(lt, lr, None, 2.0, 0.5, fp8rl.FP8RL_IS_MASK,  # noqa: E731
                                             w=w, stats=stats, loss=loss)
    elif c == "attention":
        k = wl.kv_tensor(seed=6, device=dev, seqs=64, tokens=4096)
        kq, ks = fp8rl.quantize_kv_fp8(k, fp8rl.FP8RL_KV_CALIBRATE)
        vq, vs = fp8rl.quantize_kv_fp8(k, fp8rl.FP8RL_KV_CALIBRATE)
        del k
        qh = torch.randn(64, 32, 128, device=dev).to(torch.bfloat16)
        lens = torch.full((64,), 4096, dtype=torch.int32, device=dev)
        run = lambda: fp8rl.decode_attention_fp8kv(qh, kq, vq, ks, vs, lens)  # noqa: E731
    elif c == "glue_gather":
        _, tok, _ = wl.moe_routing(seed=0)
        x = wl.dense_acts(wl.MOE_TOKENS, wl.MOE_HIDDEN, seed=7, device=dev)
        rows = tok.to(torch.int32).to(dev)
        run = lambda: fp8rl.quantize_act_gather(x, rows)  # noqa: E731
    elif c == "glue_silu":
        h = wl.expert_inputs(wl.MOE_TOKENS * wl.MOE_TOPK, 2 * wl.MOE_INTER, seed=9, device=dev)
        run = lambda: fp8rl.silu_mul_quantize(h)  # noqa: E731
    else:
        raise SystemExit("unknown case %r" % c)
    for _ in range(args.iters):
        run()
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    print("profile_case %s: %d iterations done" % (c, args.iters))


if __name__ == "__main__":
    main()
