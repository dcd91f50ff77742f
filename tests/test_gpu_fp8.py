"""FP8 expert weights (needs a GB300): the quantiser (moe_quantize_fp8) bit
for bit against the oracle's, and the FP8 layer (moe_layer_forward_fp8: the
persistent decode layer up to 16 tokens, the kernel chain with FP8 GEMMs
above) against the oracle's fp64 layer over its own dequantised weights, on
every layer configuration at decode and larger batch sizes.  The oracle
quantises the weights itself; the GPU's codes and block exponents must equal
its bytes, so both sides run the same FP8 layer."""

import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import (LayerRun, assert_output_close, bf16_np, check_routing, host_copy,
                       rel_l2, sample_tokens)
from test_gpu_layer import layer_inputs

pytestmark = pytest.mark.gpu

# relative L2 of the FP8 layer's output against the bf16 layer's, per case
FP8_QUALITY = []


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("n,rows,K,seed", [(3, 200, 448, 1), (1, 128, 128, 2), (2, 1536, 4096, 3),
                                           (5, 64, 64, 4), (2, 192, 7168, 5)])
def test_quantizer_matches_oracle(n, rows, K, seed):
    w = synth.normal((n, rows, K), seed, 1, 0.03, torch.bfloat16)
    if n >= 3:
        w[0, :5] *= 4000                    # saturation-range neighbours
        w[1, :128, :128] = 0                # an all-zero block
        w[2] = (w[2].float() * 2.0 ** -30).to(torch.bfloat16)
    wd = w.cuda()
    q = torch.empty((n, rows, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty((n, -(-rows // 128), -(-K // 128)), dtype=torch.int8, device="cuda")
    moe.moe_quantize_fp8(wd, n, rows, K, q, sc)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_fp8_c(w)
    assert np.array_equal(sc.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def _oracle_expert(w13_e, w2_e):
    """The oracle's own quantisation of one expert: dequantised bf16 W13 and
    W2, and the codes / exponents (to compare with the GPU's)."""
    I2, H = w13_e.shape
    q13, s13 = oracle.quantize_fp8_c(w13_e.reshape(2, I2 // 2, H))
    q2, s2 = oracle.quantize_fp8_c(w2_e.reshape(1, H, I2 // 2))
    d13 = oracle.dequantize_fp8(q13, s13).reshape(I2, H)
    d2 = oracle.dequantize_fp8(q2, s2).reshape(H, I2 // 2)
    return d13, d2, (q13, s13, q2, s2)


def check_fp8_layer(inputs, n_sample=None):
    cfg, T = inputs.cfg, inputs.T
    E, k, I, H = cfg.E, cfg.k, cfg.I, cfg.H
    q = moe.quantize_layer_fp8(inputs.w13, inputs.w2, inputs.w13_shared, inputs.w2_shared)
    run = LayerRun(inputs)
    wq = moe.layer_weights_fp8(inputs.w_router, q, inputs.sel_bias)
    moe.moe_layer_forward_fp8(run.d, wq, inputs.x, run.y, run.ws)
    torch.cuda.synchronize()
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, (st, raw)
    meta = run.metadata()
    host = host_copy(inputs, experts=[])
    s = oracle.router_logits(host["x"], host["w_router"])
    ids, w, gap = oracle.topk_gating(s, k, cfg.gating, host["sel_bias"])
    bias = None if host["sel_bias"] is None else host["sel_bias"].numpy()
    check_routing(meta["ids"], meta["w"], {"logits": s, "ids": ids, "w": w, "gap": gap},
                  cfg.gating, bias, label=f"{cfg.name} T={T} fp8")
    rc, ro, rp, ri = oracle.dispatch(meta["ids"], E)
    assert np.array_equal(meta["counts"], rc) and np.array_equal(meta["perm_src"], rp)
    if n_sample is None or T <= n_sample:
        toks = list(range(T))
    else:
        # tile edges of the hottest experts and of the shared expert, the
        # coldest touched expert, seeded random tokens
        toks = sample_tokens(T, n_sample, meta["ids"], rc, perm_src=meta["perm_src"],
                             offsets=meta["offsets"], shared=bool(cfg.shared))
    toks = [t for t in toks if not (gap[t] < 1e-5)]
    need = sorted({int(e) for t in toks for e in ids[t]})
    host = host_copy(inputs, experts=need)
    d13, d2 = {}, {}
    for e in need:
        d13[e], d2[e], (q13, s13, q2, s2) = _oracle_expert(host["w13"][e], host["w2"][e])
        # the GPU's bytes for this expert are the oracle's
        assert np.array_equal(q["w13"][e].cpu().numpy().reshape(q13.shape), q13)
        assert np.array_equal(q["w13_scale"][e].cpu().numpy().reshape(s13.shape), s13)
        assert np.array_equal(q["w2"][e].cpu().numpy().reshape(q2.shape), q2)
        assert np.array_equal(q["w2_scale"][e].cpu().numpy().reshape(s2.shape), s2)
    d13s = d2s = None
    if cfg.shared:
        d13s, d2s, _ = _oracle_expert(host["w13_shared"], host["w2_shared"])
    y_ref = oracle.layer_tokens(host["x"], ids, w, d13, d2, toks, d13s, d2s)
    got = bf16_np(run.y[toks])
    assert_output_close(got, y_ref, "y (fp8)")
    # the quantisation's own effect: the bf16 layer's output
    y_bf16 = oracle.layer_tokens(host["x"], ids, w, host["w13"], host["w2"], toks,
                                 host["w13_shared"], host["w2_shared"])
    FP8_QUALITY.append((f"{cfg.name} T={T}", rel_l2(y_ref, y_bf16)))
    return rel_l2(y_ref, y_bf16)


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 16), ("mixtral", 1), ("mixtral", 4),
                                    ("qwen3", 1), ("qwen3", 8), ("qwen3_tp8", 1),
                                    ("qwen3_tp8", 16), ("dsv3", 2)])
def test_fp8_layer_matches_oracle(name, T):
    q_err = check_fp8_layer(layer_inputs(name, T))
    # E4M3 with 128 x 128 block scales: a few percent of relative error against
    # the bf16 weights' layer (reported; the parity above is exact-format)
    assert q_err < 0.06


@pytest.mark.parametrize("name,T,n", [("tiny", 17, None), ("tiny", 64, None), ("mixtral", 33, None),
                                      ("qwen3", 128, 128), ("qwen3_tp8", 256, 128), ("dsv3", 32, None),
                                      ("qwen3", 1024, 96), ("mixtral", 512, 64)])
def test_fp8_chain_matches_oracle(name, T, n):
    """Batches above 16 tokens: the kernel chain with the FP8 GEMMs (fp16 token
    rows, the weight operand in TMEM), against the oracle over the same
    dequantised weights; every token up to n (sampled above, tile edges of the
    hottest and shared experts included)."""
    q_err = check_fp8_layer(layer_inputs(name, T), n_sample=n)
    assert q_err < 0.06


@pytest.mark.parametrize("T", [4, 48])
def test_fp8_values_past_fp16_range_saturate_and_flag(T):
    """h (fp16 in the FP8 layer) beyond +-65504: saturated, never inf, and the
    status word reports a device check (range bit) -- the persistent layer
    (T = 4) and the kernel chain (T = 48)."""
    cfg = synth.LayerConfig("ovf", H=256, E=4, k=2, I=256, gating=synth.GATE_TOPK_SOFTMAX)
    inp = synth.make_layer(cfg, T, 9, device="cuda")
    x = (inp.x.float() * 4000.0).to(torch.bfloat16)
    q = moe.quantize_layer_fp8(inp.w13, inp.w2)
    run = LayerRun(inp)
    moe.moe_layer_forward_fp8(run.d, moe.layer_weights_fp8(inp.w_router, q), x, run.y, run.ws)
    torch.cuda.synchronize()
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_ERR_DEVICE_CHECK and raw & (1 << 5), (st, raw)
    assert torch.isfinite(run.y.float()).all()


@pytest.mark.parametrize("name,T", [("qwen3", 8), ("mixtral", 64)])
def test_fp8_forward_replays_from_a_cuda_graph(name, T):
    """The FP8 forward (the persistent layer's cooperative launch, or the
    chain) captures into a CUDA graph; replays give the eager result bit for
    bit."""
    inp = layer_inputs(name, T)
    q = moe.quantize_layer_fp8(inp.w13, inp.w2, inp.w13_shared, inp.w2_shared)
    wq = moe.layer_weights_fp8(inp.w_router, q, inp.sel_bias)
    run = LayerRun(inp)
    moe.moe_layer_forward_fp8(run.d, wq, inp.x, run.y, run.ws)
    torch.cuda.synchronize()
    y_eager = run.y.clone()
    y = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_layer_forward_fp8(run.d, wq, inp.x, y, run.ws, stream=s)  # warm-up on s
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward_fp8(run.d, wq, inp.x, y, run.ws, stream=s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, raw
    del g
