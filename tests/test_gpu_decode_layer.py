"""The persistent single-kernel decode layer (moe_layer_forward_ex with
MOE_PATH_PERSISTENT: router, gating, dispatch, both expert GEMMs and the
combine in one cooperative launch) against the CPU oracle on every layer
configuration at decode batch sizes, and against the kernel chain on the same
inputs (needs a GB300).  Routing ids are bit-exact off near-ties, the
dispatch metadata bit-exact given the ids, outputs within the layer
tolerance."""

import numpy as np
import pytest
import torch

import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import LayerRun, assert_output_close, assert_rows_close, bf16_np
from test_gpu_layer import check_layer, layer_inputs

pytestmark = pytest.mark.gpu
PERSISTENT, CHAIN = moe.MOE_PATH_PERSISTENT, moe.MOE_PATH_KERNEL_CHAIN


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 16), ("mixtral", 1), ("mixtral", 8),
                                    ("qwen3", 1), ("qwen3", 5), ("qwen3", 16),
                                    ("qwen3_tp8", 1), ("qwen3_tp8", 2), ("qwen3_tp8", 4),
                                    ("qwen3_tp8", 16), ("dsv3", 1), ("dsv3", 16)])
def test_persistent_layer_matches_oracle(name, T):
    check_layer(layer_inputs(name, T), path=PERSISTENT)


@pytest.mark.parametrize("gating", [synth.GATE_TOPK_SOFTMAX, synth.GATE_SOFTMAX_TOPK,
                                    synth.GATE_SOFTMAX_TOPK_RENORM,
                                    synth.GATE_SIGMOID_BIAS_RENORM])
@pytest.mark.parametrize("shared", [False, True])
def test_persistent_gating_variants(gating, shared):
    cfg = synth.LayerConfig(f"pg{gating}", H=256, E=8, k=2, I=256, gating=gating, shared=shared,
                            sel_bias_std=0.1 if gating == synth.GATE_SIGMOID_BIAS_RENORM else 0.0)
    check_layer(synth.make_layer(cfg, 11, 3, device="cuda"), path=PERSISTENT)


@pytest.mark.parametrize("T,E,k,I,H", [(16, 512, 32, 128, 256),   # 512 assignments, 512 experts
                                       (3, 32, 32, 64, 256),      # every expert selected
                                       (9, 1, 1, 192, 384),       # one expert, ragged I and H
                                       (16, 32, 4, 1344, 832)])   # odd K-block counts, ragged tiles
def test_persistent_edge_shapes(T, E, k, I, H):
    cfg = synth.LayerConfig("edge", H=H, E=E, k=k, I=I, gating=synth.GATE_SOFTMAX_TOPK_RENORM)
    check_layer(synth.make_layer(cfg, T, 5, device="cuda"), path=PERSISTENT, n_sample=T)


@pytest.mark.parametrize("name,T", [("qwen3", 8), ("qwen3_tp8", 16), ("mixtral", 2)])
def test_persistent_matches_chain(name, T):
    """Both paths on the same inputs: the same experts and the same dispatch
    layout (the router logits differ only in summation order), close h and
    out_perm rows, close outputs; repeated persistent calls are bit-identical
    (its counters return to zero)."""
    inp = layer_inputs(name, T)
    cfg = inp.cfg
    a = LayerRun(inp, PERSISTENT)
    ya = a.forward().clone()
    ya2 = a.forward().clone()
    assert torch.equal(ya, ya2)
    b = LayerRun(inp, CHAIN)
    yb = b.forward().clone()
    ma, mb = a.metadata(), b.metadata()
    clear = ~(ma["gap"] < 1e-5) & ~(mb["gap"] < 1e-5)
    if clear.all():
        for key in ("ids", "counts", "offsets", "perm_src", "inv_pos"):
            assert np.array_equal(ma[key], mb[key]), key
        assert np.max(np.abs(ma["w_perm"] - mb["w_perm"])) <= 1e-5
        R = T * cfg.k
        ha = a.view("h", torch.bfloat16, (R, cfg.I)).double().cpu().numpy()
        hb = b.view("h", torch.bfloat16, (R, cfg.I)).double().cpu().numpy()
        assert_rows_close(ha, hb, "h")
        oa = a.view("out_perm", torch.float16, (R, cfg.H)).double().cpu().numpy()
        ob = b.view("out_perm", torch.float16, (R, cfg.H)).double().cpu().numpy()
        assert_rows_close(oa, ob, "out_perm")
    assert_output_close(bf16_np(ya)[clear], bf16_np(yb)[clear], "y persistent vs chain")


def test_auto_path_takes_persistent_layer_for_decode():
    """moe_layer_forward picks the persistent layer up to 16 tokens: its result
    is the persistent path's bit for bit."""
    inp = layer_inputs("qwen3_tp8", 4)
    y_auto = LayerRun(inp).forward().clone()
    y_pers = LayerRun(inp, PERSISTENT).forward().clone()
    assert torch.equal(y_auto, y_pers)
