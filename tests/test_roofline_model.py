"""Pins of the benchmark's roofline model (bench.py): the expected number of
touched experts, the bytes of one expert, the rows per expert and the
compute-bound ridge, each checked against the values the CS349D lecture 8
notes print (tests/golden/touched_experts.txt, tests/golden/per_expert_batch.txt)
and, for the touched-expert formula, against a Monte-Carlo count over the
seeded uniform routings the tests use.  The per-step byte and flop counts the
bench reports (algorithmic) are then checked on hand-made routings against
these pinned parts."""

import numpy as np
import pytest

import bench
import synth
from conftest import golden


def test_expected_touched_matches_the_printed_exercise():
    kv, rows = golden("touched_experts.txt")
    assert rows, "fixture has no rows"
    for E, k, n, want in rows:
        got = bench.expected_touched(int(E), int(k), int(n))
        places = len(want.split(".")[1]) if "." in want else 0
        assert round(got, places) == pytest.approx(float(want), abs=1e-9), (E, k, n, got)


@pytest.mark.parametrize("E,k,n", [(64, 4, 16), (128, 8, 16), (8, 2, 4), (256, 8, 8)])
def test_expected_touched_matches_monte_carlo(E, k, n):
    trials = 400
    touched = [len(np.unique(synth.random_ids(n, k, E, seed).numpy())) for seed in range(trials)]
    mean, sd = float(np.mean(touched)), float(np.std(touched))
    want = bench.expected_touched(E, k, n)
    # mean of 400 samples: standard error sd / 20; allow 4 standard errors
    assert abs(mean - want) <= 4 * sd / np.sqrt(trials) + 1e-9, (mean, want, sd)


def test_expected_touched_limits():
    assert bench.expected_touched(128, 8, 1) == pytest.approx(8)
    assert bench.expected_touched(128, 8, 100000) == pytest.approx(128)
    assert bench.expected_touched(8, 8, 1) == pytest.approx(8)


def test_mixtral_expert_size_matches_the_page():
    kv, _ = golden("touched_experts.txt")
    params = bench.expert_params(4096, 14336)
    assert params == 176_160_768
    assert round(params / 1e8, 2) == float(kv["expert_params_mixtral"][0]) / 1e8
    b = bench.expert_bytes(4096, 14336)
    assert b == 352_321_536
    assert round(b / 1e9, 2) == float(kv["expert_gb_bf16_mixtral"][0])


def test_rows_per_expert_and_ridge_match_the_page():
    kv, rows = golden("per_expert_batch.txt")
    for n, k, E, want in rows:
        assert bench.tokens_per_expert(int(n), int(k), int(E)) == float(want)
    # A100: 312 TFLOPS over 2 TB/s -> 156 rows per expert; Qwen3-235B (128
    # experts, top-8) then needs 156 * 128 / 8 = 2496 tokens per batch
    ridge = bench.ridge_rows(312e12, 2e12)
    assert ridge == float(kv["ridge_a100_tokens"][0])
    assert ridge * 128 / 8 == float(kv["batch_for_compute_bound_qwen3_a100"][0])
    # a batch of 400 gives 25 rows per expert: 16% of the tensor peak
    util = bench.expert_gemm_utilisation(bench.tokens_per_expert(400, 8, 128), 312e12, 2e12)
    assert round(100 * util) == float(kv["utilisation_batch400_percent"][0])


def test_expert_intensity_is_rows_per_expert():
    # the ridge reasoning: an expert with m rows does 2 * m * params flops over
    # 2 * params bytes, so flops per byte = m
    cfg = synth.CONFIGS["qwen3"]
    for m in (1, 25, 156):
        flops = 2 * m * bench.expert_params(cfg.H, cfg.I)
        assert flops / bench.expert_bytes(cfg.H, cfg.I) == m


def test_algorithmic_counts_touched_experts_and_activations():
    cfg = synth.CONFIGS["qwen3"]
    T = 16
    counts = [0] * cfg.E
    for e in range(16):              # 16 experts, 8 rows each: T * k = 128
        counts[e * 3] = 8
    a = bench.algorithmic(cfg, T, counts)
    assert a["touched"] == 16
    weights = 16 * bench.expert_bytes(cfg.H, cfg.I)
    router = cfg.E * cfg.H * 4
    xy = 2 * T * cfg.H * 2
    assert a["layer_bytes"] == weights + router + xy
    # flops: every assignment runs one expert (2 flops per multiply-add), plus
    # the fp32 router
    assert a["layer_flops"] == 2 * T * cfg.k * bench.expert_params(cfg.H, cfg.I) + 2 * T * cfg.H * cfg.E
    # the same routing with one more expert touched adds exactly one expert's bytes
    counts[1] = 1
    b = bench.algorithmic(cfg, T, counts)
    assert b["layer_bytes"] - a["layer_bytes"] == bench.expert_bytes(cfg.H, cfg.I)


def test_algorithmic_shared_expert_adds_one_expert_for_every_token():
    cfg = synth.CONFIGS["dsv3"]
    T = 32
    counts = [1] * cfg.E
    a = bench.algorithmic(cfg, T, counts)
    per = bench.expert_bytes(cfg.H, cfg.I)
    assert a["layer_bytes"] == (cfg.E + 1) * per + cfg.E * cfg.H * 4 + 2 * T * cfg.H * 2
    routed = 2 * T * cfg.k * bench.expert_params(cfg.H, cfg.I)
    shared = 2 * T * bench.expert_params(cfg.H, cfg.I)
    assert a["layer_flops"] == routed + shared + 2 * T * cfg.H * cfg.E
