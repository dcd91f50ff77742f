"""The expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2), which the kernel
chain takes for prefill batches (T*k >= 256*E; H a multiple of 256, I of 128):
parity with the oracle on every token of small layers that reach the pair
tiles (ragged expert segments, token chunks that end inside a 256-row tile,
segments shorter than one tile, the shared expert, output widths of 1 to 3
pair tiles), agreement with the one-SM chain on the same inputs, and a check
that the pair kernels are the ones that ran (needs a GB300)."""

import numpy as np
import pytest
import torch

import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import LayerRun, bf16_np, rel_l2
from test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    torch.cuda.empty_cache()


# (name, T, H, E, k, I, gating, shared, skew): T*k >= 256*E (both GEMMs on
# pairs) except pair_down, whose down GEMM alone takes pairs (I >= 2048 with
# 64 <= T*k/E < 256)
CASES = [
    ("pair_min", 512, 256, 4, 2, 128, synth.GATE_TOPK_SOFTMAX, False, None),
    ("pair_down", 256, 256, 4, 2, 2048, synth.GATE_TOPK_SOFTMAX, True, ("normal", 0.5)),
    ("pair_skew", 700, 512, 4, 2, 256, synth.GATE_SIGMOID_BIAS_RENORM, True, ("normal", 1.0)),
    ("pair_wide", 300, 768, 2, 2, 384, synth.GATE_SOFTMAX_TOPK_RENORM, True, None),
    ("pair_mid", 2048, 1024, 8, 2, 512, synth.GATE_SOFTMAX_TOPK, False, ("normal", 0.5)),
]


def inputs(name, T, H, E, k, I, gating, shared, skew, seed=5):
    cfg = synth.LayerConfig(name, H=H, E=E, k=k, I=I, gating=gating, shared=shared, skew=skew,
                            sel_bias_std=0.1 if gating == synth.GATE_SIGMOID_BIAS_RENORM else 0.0)
    return synth.make_layer(cfg, T, seed, device="cuda")


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pair_layer_matches_oracle(case):
    inp = inputs(*case)
    info = check_layer(inp, n_sample=min(inp.T, 512))
    assert info["checked_tokens"] >= min(inp.T, 512) - 8  # near-ties aside


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pair_matches_one_sm_chain(case):
    inp = inputs(*case)
    y_pair = LayerRun(inp).forward().clone()
    y_one = LayerRun(inp, moe.MOE_PATH_CHAIN_ONE_SM).forward()
    a, b = bf16_np(y_pair), bf16_np(y_one)
    # the same products accumulated in the same K order: equal up to the
    # rounding of fp32 partial sums
    assert rel_l2(a, b) <= 1e-3, rel_l2(a, b)


def test_pair_kernels_run():
    """The profiler's kernel list of one prefill forward holds the pair
    kernels and not the one-SM GEMM; the one-SM path holds the reverse."""
    prof_mod = pytest.importorskip("torch.profiler")
    inp = inputs(*CASES[3])

    def kernels(path):
        run = LayerRun(inp, path)
        run.forward()
        try:
            with prof_mod.profile(activities=[prof_mod.ProfilerActivity.CUDA]) as prof:
                run.forward()
        except Exception as exc:  # no CUPTI on this host
            pytest.skip(f"profiler unavailable: {exc}")
        return {e.name for e in prof.events()}

    names = kernels(None)
    if not names:
        pytest.skip("the profiler recorded no kernels")
    assert any("expert_gemm_pair_kernel" in n for n in names), sorted(names)
    assert not any("expert_gemm_kernel" in n for n in names), sorted(names)
    names = kernels(moe.MOE_PATH_CHAIN_ONE_SM)
    assert not any("expert_gemm_pair_kernel" in n for n in names), sorted(names)
    assert any("expert_gemm_kernel" in n for n in names), sorted(names)


def test_pair_path_graph_replay():
    inp = inputs(*CASES[1])
    run = LayerRun(inp)
    y_eager = run.forward().clone()
    y = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_layer_forward(run.d, run.w, inp.x, y, run.ws, stream=s)  # warm-up on s
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward(run.d, run.w, inp.x, y, run.ws, stream=s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
    st, raw = moe.moe_get_device_status(run.ws)
    assert st == moe.MOE_OK, raw
    del g
