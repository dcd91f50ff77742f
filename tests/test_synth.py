"""The seeded input generator: determinism, distribution, workload recipe."""

import math

import numpy as np
import pytest
import torch

import oracle
import synth


def test_counter_generator_is_deterministic_and_sliceable():
    a = synth.normal((1000,), 0, 4, 1.0, torch.float32)
    b = synth.normal((1000,), 0, 4, 1.0, torch.float32)
    assert torch.equal(a, b)
    tail = torch.empty(300, dtype=torch.float32)
    synth.normal_(tail, 0, 4, 1.0, start=700)
    assert torch.equal(tail, a[700:])
    assert not torch.equal(a, synth.normal((1000,), 1, 4, 1.0, torch.float32))
    assert not torch.equal(a, synth.normal((1000,), 0, 5, 1.0, torch.float32))


def test_counter_generator_moments():
    z = synth.normal((1 << 20,), 0, 1, 1.0, torch.float64).numpy()
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    # tail mass of a standard normal: P(|z| > 2) = 0.0455
    assert abs((np.abs(z) > 2).mean() - 0.0455) < 2e-3


def test_hash_matches_reference_integer_arithmetic():
    # The tensor path (16-bit split multiplies) equals plain modular arithmetic.
    v = torch.tensor([0, 1, 12345, 0xFFFFFFFF, 0x80000000], dtype=torch.int64)
    got = synth._hash32(v).tolist()
    assert got == [synth._hash32_int(int(t)) for t in v]


def test_layer_shapes_and_scales():
    inp = synth.make_layer(synth.CONFIGS["tiny"], 64, seed=0)
    cfg = inp.cfg
    assert inp.x.shape == (64, cfg.H) and inp.x.dtype == torch.bfloat16
    assert inp.w_router.shape == (cfg.E, cfg.H) and inp.w_router.dtype == torch.float32
    assert inp.w13.shape == (cfg.E, 2 * cfg.I, cfg.H) and inp.w2.shape == (cfg.E, cfg.H, cfg.I)
    assert abs(inp.w13.float().std().item() - cfg.H ** -0.5) < 2e-3
    assert abs(inp.w2.float().std().item() - cfg.I ** -0.5) < 2e-3
    assert abs(inp.w_router.std().item() - 0.02) < 1e-3
    assert inp.sel_bias is None and inp.w13_shared is None


def test_skew_channel_and_offsets():
    cfg = synth.CONFIGS["mixtral"]
    x = synth.make_tokens(cfg, 4, 0)
    assert torch.all(x[:, 0] == 1.0)
    w_r, b = synth.make_router(cfg, 0)
    delta = synth.logit_offsets(cfg, 0)
    assert np.array_equal(w_r[:, 0].numpy(), np.array(delta, dtype=np.float32))
    z = synth.logit_offsets(synth.CONFIGS["dsv3"], 0)
    assert max(z) == 0.0 and min(z) == pytest.approx(-1.2 * math.log(256))
    assert sorted(z, reverse=True)[1] == pytest.approx(-1.2 * math.log(2))


def test_qwen3_zipf_skew_hits_imbalance_target():
    # The configuration asks for an imbalance ratio of about 3 at T=1024.
    cfg = synth.CONFIGS["qwen3"]
    x = synth.make_tokens(cfg, 1024, 0)
    w_r, _ = synth.make_router(cfg, 0)
    s = oracle.router_logits(x, w_r)
    ids, _, _ = oracle.topk_gating(s, cfg.k, cfg.gating)
    counts, _, _, _ = oracle.dispatch(ids, cfg.E)
    num, den = oracle.imbalance(counts, ids.size)
    assert 2.7 <= num / den <= 3.3


def test_random_ids_distinct_per_token():
    ids = synth.random_ids(200, 8, 64, 0).numpy()
    assert all(len(set(r)) == 8 for r in ids)
    assert ids.min() >= 0 and ids.max() < 64
    hot = synth.skewed_ids(50, 4, 16, 0, hot=3).numpy()
    assert all(3 in r and len(set(r)) == 4 for r in hot)
