"""Failure reporting without a GPU fault (needs a GB300 for the GPU tests).

The pipelined kernels bound every wait and report a wait that ran out in the
workspace status word instead of hanging.  moe_check_bounded_wait makes one
such wait run out -- a barrier that nothing completes -- and the test checks
that the host reads MOE_ERR_TIMEOUT with the check's bit, that clearing the
word works, and that the same context then still computes a correct layer.
moe_check_bounded_grid_wait does the same for the persistent decode layer's
grid barrier (a barrier sized for more CTAs than the launch has)."""

import pytest
import torch

import routed_expert_ffn_gb300 as moe
from gpu_check import LayerRun
from test_gpu_layer import check_layer, layer_inputs


@pytest.mark.gpu
def test_bounded_wait_reports_and_context_survives():
    from routed_expert_ffn_gb300 import build
    build.build()
    d = moe.desc(64, 256, 8, 2, 512, moe.MOE_GATE_TOPK_SOFTMAX)
    ws = moe.alloc_workspace(d)
    moe.moe_check_bounded_wait(ws)
    st, raw = moe.moe_get_device_status(ws, clear=True)
    assert st == moe.MOE_ERR_TIMEOUT and raw & (1 << 6), (st, raw)
    st, raw = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK and raw == 0
    torch.cuda.synchronize()
    check_layer(layer_inputs("tiny", 64), n_sample=16)


@pytest.mark.gpu
def test_bounded_grid_wait_reports_and_context_survives():
    from routed_expert_ffn_gb300 import build
    build.build()
    d = moe.desc(4, 256, 8, 2, 512, moe.MOE_GATE_TOPK_SOFTMAX)
    ws = moe.alloc_workspace(d)
    moe.moe_check_bounded_grid_wait(ws)
    st, raw = moe.moe_get_device_status(ws, clear=False)
    assert st == moe.MOE_ERR_TIMEOUT and raw & (1 << 7), (st, raw)
    # the barrier's arrival count is left behind: re-initialise the workspace
    moe.moe_workspace_init(ws)
    st, raw = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK and raw == 0
    torch.cuda.synchronize()
    # the same workspace then runs the persistent layer: equal to a fresh
    # workspace's result bit for bit, and that result matches the oracle
    inp = layer_inputs("tiny", 4)
    fresh = LayerRun(inp, moe.MOE_PATH_PERSISTENT)
    y_ref = fresh.forward().clone()
    reused = LayerRun(inp, moe.MOE_PATH_PERSISTENT)
    reused.ws = ws
    assert torch.equal(reused.forward(), y_ref)
    check_layer(inp, path=moe.MOE_PATH_PERSISTENT)
