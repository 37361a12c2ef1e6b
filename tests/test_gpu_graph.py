"""The hot path captured in a CUDA graph: serving engines capture their
decode steps, so every stream-ordered entry point must be capturable once the
library has seen the device.  One step's calls (whole-model multi-tensor
re-quantization, activation quantization, dense GEMMs of both flavours,
gather, grouped GEMM, SiLU glue, KV calibrate and quantize, decode attention,
TIS, IS statistics with the weighted loss) are run eagerly, then captured and
replayed into separate outputs; the results must agree bit for bit, except
the statistics sums, whose FP64 atomic order may differ (counts stay exact).
The replayed outputs are also checked against the oracle directly: codes,
scales and weights bit for bit, the GEMMs and the attention within their
tolerances."""
import numpy as np
import pytest
import torch

import fp8_precision_rollout_gb300 as fp8rl
import oracle
from fp8_precision_rollout_gb300 import workloads
from gpu_helpers import check_gemm, device, np_f32_bits, np_u8

pytestmark = pytest.mark.gpu


def _inputs(dev):
    g = torch.Generator().manual_seed(11)
    inp = {}
    inp["ws"] = [workloads.make_weight(n, k, seed=100 + i, device=dev)
                 for i, (n, k) in enumerate(((2048, 1024), (256, 256), (1024, 768)))]
    inp["a_pre"] = workloads.dense_acts(1280, 1024, seed=3, device=dev)    # 80 tiles: one CTA each
    inp["a_dec"] = workloads.dense_acts(64, 1024, seed=4, device=dev)      # split-K flavour
    inp["tok"] = workloads.dense_acts(96, 256, seed=5, device=dev)
    counts = torch.tensor([40, 0, 130, 7, 300, 5], dtype=torch.int64)
    offs = torch.zeros(7, dtype=torch.int32)
    offs[1:] = torch.cumsum(counts, 0).to(torch.int32)
    inp["offsets"] = offs.to(dev)
    inp["rows"] = torch.randint(0, 96, (int(counts.sum()),), generator=g, dtype=torch.int32).to(dev)
    inp["we"] = workloads.make_weight(6 * 512, 256, seed=7, device=dev)     # 6 experts [512, 256]
    inp["kv"] = workloads.kv_tensor(seed=8, device=dev, seqs=3, tokens=700, heads=2)
    inp["q"] = torch.randn(3, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    inp["lens"] = torch.tensor([700, 1, 333], dtype=torch.int32, device=dev)
    lt, lr = workloads.tis_logprobs(10007, seed=9, device=dev)
    inp["lt"], inp["lr"] = lt, lr
    inp["loss"] = torch.randn(10007, generator=g).to(dev)
    return inp


def _outputs(inp, dev):
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    o = {}
    o["wq"] = [torch.empty(w.shape, dtype=u8, device=dev) for w in inp["ws"]]
    o["wsc"] = [torch.empty((w.shape[0] + 127) // 128, (w.shape[1] + 127) // 128, dtype=f32,
                            device=dev) for w in inp["ws"]]
    o["ap_q"] = torch.empty(1280, 1024, dtype=u8, device=dev)
    o["ap_s"] = torch.empty(8, 1280, dtype=f32, device=dev)
    o["ad_q"] = torch.empty(64, 1024, dtype=u8, device=dev)
    o["ad_s"] = torch.empty(8, 64, dtype=f32, device=dev)
    o["y_pre"] = torch.empty(1280, 2048, dtype=bf, device=dev)
    o["y_dec"] = torch.empty(64, 2048, dtype=bf, device=dev)
    m = int(inp["rows"].numel())
    o["g_q"] = torch.empty(m, 256, dtype=u8, device=dev)
    o["g_s"] = torch.empty(2, m, dtype=f32, device=dev)
    o["weq"] = torch.empty(6 * 512, 256, dtype=u8, device=dev)
    o["wes"] = torch.empty(6 * 4, 2, dtype=f32, device=dev)
    o["h"] = torch.empty(m, 512, dtype=bf, device=dev)
    o["s_q"] = torch.empty(m, 256, dtype=u8, device=dev)
    o["s_s"] = torch.empty(2, m, dtype=f32, device=dev)
    o["kq"] = torch.empty(inp["kv"].shape, dtype=u8, device=dev)
    o["ks"] = torch.empty(2, dtype=f32, device=dev)
    o["att"] = torch.empty(3, 8, 128, dtype=bf, device=dev)
    o["tw"] = torch.empty(10007, dtype=f32, device=dev)
    o["mw"] = torch.empty(10007, dtype=f32, device=dev)
    o["st"] = torch.empty(6, dtype=torch.float64, device=dev)
    return o


def _step(inp, o):
    fp8rl.quantize_weights_blockwise_multi(inp["ws"], o["wq"], o["wsc"])
    fp8rl.quantize_act_groupwise(inp["a_pre"], o["ap_q"], o["ap_s"])
    fp8rl.gemm_w8a8_blockwise(o["ap_q"], o["ap_s"], o["wq"][0], o["wsc"][0], o["y_pre"])
    fp8rl.quantize_act_groupwise(inp["a_dec"], o["ad_q"], o["ad_s"])
    fp8rl.gemm_w8a8_blockwise(o["ad_q"], o["ad_s"], o["wq"][0], o["wsc"][0], o["y_dec"])
    fp8rl.quantize_act_gather(inp["tok"], inp["rows"], o["g_q"], o["g_s"])
    fp8rl.quantize_weights_blockwise(inp["we"], o["weq"], o["wes"])
    fp8rl.grouped_gemm_w8a8_blockwise(o["g_q"], o["g_s"], o["weq"].view(6, 512, 256),
                                      o["wes"].view(6, 4, 2), inp["offsets"], o["h"])
    fp8rl.silu_mul_quantize(o["h"], o["s_q"], o["s_s"])
    fp8rl.quantize_kv_fp8(inp["kv"], fp8rl.FP8RL_KV_CALIBRATE, o["ks"], o["kq"])
    fp8rl.decode_attention_fp8kv(inp["q"], o["kq"], o["kq"], o["ks"], o["ks"], inp["lens"],
                                 out=o["att"])
    fp8rl.tis_weights(inp["lt"], inp["lr"], None, 2.0, 0.0, o["tw"])
    fp8rl.is_weights_stats(inp["lt"], inp["lr"], None, 2.0, 0.5, fp8rl.FP8RL_IS_MASK, w=o["mw"],
                           stats=o["st"], loss=inp["loss"])


def test_step_replays_from_a_cuda_graph():
    dev = device()
    inp = _inputs(dev)
    eager = _outputs(inp, dev)
    _step(inp, eager)                       # also creates the library's device state
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    graph_out = _outputs(inp, dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(inp, graph_out)               # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in graph_out.values():
        for x in (t if isinstance(t, list) else [t]):
            x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(inp, graph_out)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    for key, a in eager.items():
        b = graph_out[key]
        pairs = list(zip(a, b)) if isinstance(a, list) else [(a, b)]
        for x, y in pairs:
            if key == "st":
                assert x[0] == y[0] and x[4] == y[4], key          # counts exact
                assert torch.allclose(x, y, rtol=1e-6, atol=1e-9), key
            else:
                assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), key


def _check_against_oracle(inp, o):
    for w, q, sc in zip(inp["ws"], o["wq"], o["wsc"]):
        oq, os_ = oracle.quantize_weights_blockwise(w.cpu())
        assert (np_u8(q) == oq).all() and (np_f32_bits(sc) == os_.view(np.uint32)).all()
    for a, key in ((inp["a_pre"], "ap"), (inp["a_dec"], "ad")):
        oq, os_ = oracle.quantize_act_groupwise(a.cpu())
        assert (np_u8(o[key + "_q"]) == oq).all()
        assert (np_f32_bits(o[key + "_s"]) == os_.view(np.uint32)).all()
    w0q, w0s = np_u8(o["wq"][0]), o["wsc"][0].cpu().numpy()
    rows = np.arange(0, 1280, 7)
    y64, ab = oracle.gemm_w8a8(np_u8(o["ap_q"]), o["ap_s"].cpu().numpy(), w0q, w0s, rows=rows)
    check_gemm(o["y_pre"][torch.from_numpy(rows).to(o["y_pre"].device)], y64, ab, "graph prefill")
    y64, ab = oracle.gemm_w8a8(np_u8(o["ad_q"]), o["ad_s"].cpu().numpy(), w0q, w0s)
    check_gemm(o["y_dec"], y64, ab, "graph decode")
    oq, os_ = oracle.quantize_act_gather(inp["tok"].cpu(), inp["rows"].cpu().numpy())
    assert (np_u8(o["g_q"]) == oq).all() and (np_f32_bits(o["g_s"]) == os_.view(np.uint32)).all()
    oq, os_ = oracle.silu_mul_quantize(o["h"].cpu())
    assert (np_u8(o["s_q"]) == oq).all() and (np_f32_bits(o["s_s"]) == os_.view(np.uint32)).all()
    kv = inp["kv"].view(-1, 2, 128).cpu()
    os_ = oracle.kv_calibrate(kv)
    assert (np_f32_bits(o["ks"]) == os_.view(np.uint32)).all()
    assert (np_u8(o["kq"]).reshape(-1, 2, 128) == oracle.kv_quantize(kv, os_)).all()
    ow = oracle.tis_weights(inp["lt"].cpu().numpy(), inp["lr"].cpu().numpy())
    assert (np_f32_bits(o["tw"]) == ow.view(np.uint32)).all()
    mw, st, ta = oracle.is_weights_stats(inp["lt"].cpu().numpy(), inp["lr"].cpu().numpy(), None,
                                         2.0, 0.5, oracle.IS_MASK, inp["loss"].cpu().numpy())
    assert (np_f32_bits(o["mw"]) == mw.view(np.uint32)).all()
    got = o["st"].cpu().numpy()
    assert got[0] == st[0] and got[4] == st[4]
    assert (np.abs(got - st) <= 2.0 ** -20 * ta + 1e-300).all()
    kq = np_u8(o["kq"]).reshape(3, 700, 2, 128)
    o64, mag = oracle.decode_attention_fp8kv(inp["q"].cpu(), kq, kq, o["ks"].cpu().numpy(),
                                             o["ks"].cpu().numpy(), [700, 1, 333])
    ag = o["att"].float().cpu().numpy().astype(np.float64)
    assert (np.abs(ag - o64) <= 2.0 ** -8 * np.abs(o64) + 1e-3 * mag + 1e-30).all()


def test_graph_replay_matches_the_oracle():
    dev = device()
    inp = _inputs(dev)
    warm = _outputs(inp, dev)
    _step(inp, warm)
    torch.cuda.synchronize()
    out = _outputs(inp, dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(inp, out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in out.values():
        for x in (t if isinstance(t, list) else [t]):
            x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(inp, out)
    g.replay()
    torch.cuda.synchronize()
    fp8rl.device_status(0)
    _check_against_oracle(inp, out)
