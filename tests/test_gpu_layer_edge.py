"""Whole-layer parity with the CPU oracle on the shapes the five layer
configurations do not reach (needs a GB300): every gating variant with and
without a shared expert on both router paths (up to 32 tokens: the
one-launch router; more: the tensor-core router), the widest fan-out the
library accepts (E = 512, k = 32), every expert selected (k = E), a single
routed expert, and the standalone stage calls against the fused forward."""

import numpy as np
import pytest
import torch

import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import LayerRun
from test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    torch.cuda.empty_cache()


def inputs(name, T, H, E, k, I, gating, shared=False, skew=None, seed=3):
    cfg = synth.LayerConfig(name, H=H, E=E, k=k, I=I, gating=gating, shared=shared, skew=skew,
                            sel_bias_std=0.1 if gating == synth.GATE_SIGMOID_BIAS_RENORM else 0.0)
    return synth.make_layer(cfg, T, seed, device="cuda")


@pytest.mark.parametrize("gating", [synth.GATE_TOPK_SOFTMAX, synth.GATE_SOFTMAX_TOPK,
                                    synth.GATE_SOFTMAX_TOPK_RENORM,
                                    synth.GATE_SIGMOID_BIAS_RENORM])
@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("T", [1, 40])
def test_gating_variants(gating, shared, T):
    check_layer(inputs(f"g{gating}", T, 256, 8, 2, 256, gating, shared), n_sample=64)


@pytest.mark.parametrize("T", [3, 40])
def test_widest_fan_out(T):
    # 512 experts, 32 per token: a segment per expert, most of them tiny
    check_layer(inputs("fan", T, 256, 512, 32, 128, synth.GATE_SOFTMAX_TOPK_RENORM), n_sample=48)


def test_every_expert_selected():
    check_layer(inputs("all", 33, 256, 8, 8, 256, synth.GATE_TOPK_SOFTMAX), n_sample=48)


def test_single_routed_expert_with_shared():
    check_layer(inputs("one", 50, 256, 1, 1, 256, synth.GATE_TOPK_SOFTMAX, shared=True),
                n_sample=50)


@pytest.mark.parametrize("T", [7, 100])
def test_stage_calls_match_layer_forward(T):
    """moe_route -> moe_build_dispatch -> moe_grouped_swiglu_ffn -> moe_combine
    produces exactly the fused forward's routing and output."""
    inp = inputs("chain", T, 512, 16, 4, 256, synth.GATE_SOFTMAX_TOPK_RENORM,
                 skew=("zipf", 1.1, 0.3))
    cfg = inp.cfg
    # the kernel chain: the stage calls below are its stages
    run = LayerRun(inp, moe.MOE_PATH_KERNEL_CHAIN)
    y_fused = run.forward().clone()
    meta = run.metadata()

    d = run.d
    ws = moe.alloc_workspace(d)
    E, k = cfg.E, cfg.k
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    gap = torch.empty((T,), dtype=torch.float32, device="cuda")
    moe.moe_route(d, inp.x, inp.w_router, inp.sel_bias, logits, ids, w, gap, ws)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    wp = torch.empty(T * k, dtype=torch.float32, device="cuda")
    moe.moe_build_dispatch(d, ids, w, counts, offsets, perm, inv, wp, ws)
    out = torch.empty((T * k, cfg.H), dtype=torch.float16, device="cuda")
    moe.moe_grouped_swiglu_ffn(d, inp.x, perm, offsets, wp, inp.w13, inp.w2, None, None, out, ws)
    y = torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(d, out, inv, None, y)
    torch.cuda.synchronize()
    st, raw = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK, raw
    assert np.array_equal(ids.cpu().numpy(), meta["ids"])
    assert np.array_equal(w.cpu().numpy(), meta["w"])
    assert np.array_equal(perm.cpu().numpy(), meta["perm_src"])
    assert torch.equal(y, y_fused)


@pytest.mark.parametrize("name,T,path", [("qwen3", 1, None), ("qwen3", 1, 1), ("qwen3", 300, None),
                                         ("qwen3_tp8", 8, 2)])
def test_layer_forward_replays_from_a_cuda_graph(name, T, path):
    """The forward makes no host synchronisation or host-side decision on
    device data, so it can be captured in a CUDA graph (the persistent decode
    layer's cooperative launch included); replays give exactly the eager
    result (and leave the split-K, router, barrier and readiness counters at
    zero)."""
    cfg = synth.CONFIGS[name]
    inp = synth.make_layer(cfg, T, 0, device="cuda")
    run = LayerRun(inp, path)
    y_eager = run.forward().clone()
    y = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_layer_forward(run.d, run.w, inp.x, y, run.ws, stream=s, path=path)  # warm-up on s
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward(run.d, run.w, inp.x, y, run.ws, stream=s, path=path)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, raw
    del g
