"""The capacity-limited layer forward (moe_layer_forward_capacity) against the
oracle's capacity dispatch and layer ("MoE推理优化全景指南", "Capacity、padding
与 token dropping": C = ceil(cf x N_a / E), assignments beyond C dropped; a
dropped pair contributes 0).  Needs a GB300.  The kept layout is compared bit
for bit with the oracle's capacity dispatch of the GPU's own expert ids, the
outputs within the layer tolerance on every token up to 256 tokens (dropped
assignments included), a capacity that never binds reproduces the dropless
kernel chain bit for bit, and the call replays from a CUDA graph."""

import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import LayerRun, assert_output_close, bf16_np, check_routing, host_copy, sample_tokens
from test_gpu_layer import layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_capacity(inputs, C):
    run = LayerRun(inputs)
    moe.moe_layer_forward_capacity(run.d, run.w, inputs.x, run.y, C, run.ws)
    torch.cuda.synchronize()
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, (st, raw)
    return run


def check_capacity(inputs, cf, n_sample=256):
    cfg, T = inputs.cfg, inputs.T
    E, k = cfg.E, cfg.k
    C = moe.moe_expert_capacity(cf, T, k, E)
    assert C == oracle.expert_capacity(*_frac(cf), T * k, E)
    run = run_capacity(inputs, C)
    meta = run.metadata()
    host = host_copy(inputs, experts=[])
    s = oracle.router_logits(host["x"], host["w_router"])
    ids, w, gap = oracle.topk_gating(s, k, cfg.gating, host["sel_bias"])
    bias = None if host["sel_bias"] is None else host["sel_bias"].numpy()
    check_routing(meta["ids"], meta["w"], {"logits": s, "ids": ids, "w": w, "gap": gap},
                  cfg.gating, bias, label=f"{cfg.name} T={T} capacity {C}")
    # the kept layout of the GPU's ids, bit for bit
    kc, ko, kp, ki = oracle.capacity_dispatch(meta["ids"], E, C)
    n_kept = int(ko[E])
    assert np.array_equal(meta["counts"], kc)
    assert np.array_equal(meta["offsets"], ko)
    assert np.array_equal(meta["perm_src"][:n_kept], kp)
    assert np.all(meta["perm_src"][n_kept:] == -1)
    assert np.array_equal(meta["inv_pos"], ki)
    assert np.array_equal(meta["w_perm"][:n_kept], meta["w"].reshape(-1)[kp])
    dropped = int(np.sum(ki < 0))
    # outputs: the oracle layer with the dropped pairs' weights set to 0
    # (GPU ids and gate weights, themselves checked above)
    toks = sample_tokens(T, n_sample, meta["ids"], meta["counts"])
    drop_tok = sorted({int(a) // k for a in np.where(ki < 0)[0]})
    toks = sorted(set(toks) | set(drop_tok[:32]))
    wk = oracle.kept_weights(meta["ids"], meta["w"].astype(np.float64), E, C)
    need = sorted({int(e) for t in toks for e in meta["ids"][t]})
    host = host_copy(inputs, experts=need)
    y_ref = oracle.layer_tokens(host["x"], meta["ids"], wk, host["w13"], host["w2"], toks,
                                host["w13_shared"], host["w2_shared"])
    assert_output_close(bf16_np(run.y[toks]), y_ref, "y (capacity)")
    return C, dropped


def _frac(cf):
    from fractions import Fraction
    f = Fraction(cf).limit_denominator(10 ** 6)
    return f.numerator, f.denominator


@pytest.mark.parametrize("name,T,cf", [("tiny", 64, 1.25), ("qwen3", 256, 1.0),
                                       ("mixtral", 64, 1.0), ("qwen3_tp8", 2048, 1.25),
                                       ("dsv3", 1024, 1.0), ("dsv3", 64, 0.5)])
def test_capacity_layer_matches_oracle(name, T, cf):
    C, dropped = check_capacity(layer_inputs(name, T), cf)
    if name in ("qwen3", "dsv3"):   # skewed routing: the limit binds
        assert dropped > 0


def test_capacity_that_never_binds_is_the_dropless_chain():
    inp = layer_inputs("qwen3", 200)
    y_chain = LayerRun(inp, moe.MOE_PATH_KERNEL_CHAIN).forward().clone()
    run = run_capacity(inp, inp.T * inp.cfg.k)
    assert torch.equal(run.y, y_chain)
    assert np.all(run.metadata()["inv_pos"] >= 0)


def test_capacity_layer_replays_from_a_cuda_graph():
    inp = layer_inputs("qwen3", 300)
    C = moe.moe_expert_capacity(1.0, 300, 8, 128)
    run = run_capacity(inp, C)
    y_eager = run.y.clone()
    y = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_layer_forward_capacity(run.d, run.w, inp.x, y, C, run.ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward_capacity(run.d, run.w, inp.x, y, C, run.ws, stream=s)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, raw
    del g


@pytest.mark.parametrize("name,T,cf", [("qwen3", 16, 1.25), ("qwen3_tp8", 8, 1.0),
                                       ("mixtral", 8, 0.5)])
def test_capacity_layer_small_batches(name, T, cf):
    # tiny capacities leave most permuted rows unused: the GEMM tiles' extra
    # token columns read never-written rows, which must not matter
    check_capacity(layer_inputs(name, T), cf)
