"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to what the pages or the mathematics fix:
the pages' worked examples (tests/golden), closed forms, invariants, special
cases that reduce to a library routine, and brute force on tiny inputs.  A
plausible slip in the oracle (wrong sign, swapped gate/up, transposed W2,
dropped shared expert, wrong tie-break, bias leaking into the weights, wrong
segment order) fails at least one of them.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden

MODES = [oracle.GATE_TOPK_SOFTMAX, oracle.GATE_SOFTMAX_TOPK, oracle.GATE_SOFTMAX_TOPK_RENORM,
         oracle.GATE_SIGMOID_BIAS_RENORM]


def _inject_scores(scores, H=256, seed=3):
    """x = e_0 (bf16 1.0), W_r[:,0] = scores: the router's fp32 logits are then
    exactly fp32(scores) (every other product is zero)."""
    E = len(scores)
    x = torch.zeros((1, H), dtype=torch.bfloat16)
    x[0, 0] = 1.0
    w_r = synth.normal((E, H), seed, 99, 0.5, torch.float32)
    w_r[:, 0] = torch.tensor(scores, dtype=torch.float32)
    return x, w_r


# ----------------------------------------------------------------- routing --

def test_router_logits_exact_on_injected_scores():
    kv, _ = golden("router_8expert_top2.txt")
    scores = [float(v) for v in kv["scores"]]
    x, w_r = _inject_scores(scores)
    s = oracle.router_logits(x, w_r)
    assert np.array_equal(s[0], np.array(scores, dtype=np.float32))


@pytest.mark.parametrize("mode", MODES)
def test_page_example_selects_experts_1_and_4(mode):
    kv, _ = golden("router_8expert_top2.txt")
    scores = [float(v) for v in kv["scores"]]
    k = int(kv["k"][0])
    x, w_r = _inject_scores(scores)
    s = oracle.router_logits(x, w_r)
    bias = np.zeros(len(scores), dtype=np.float32)
    ids, w, gap = oracle.topk_gating(s, k, mode, bias)
    assert ids[0].tolist() == [int(v) for v in kv["selected"]]
    assert gap[0] > 0


def test_topk_softmax_weights_closed_form_on_page_example():
    # Two kept logits a > b: softmax gives (sigmoid(a-b), sigmoid(b-a)).
    kv, _ = golden("router_8expert_top2.txt")
    scores = [float(v) for v in kv["scores"]]
    x, w_r = _inject_scores(scores)
    s = oracle.router_logits(x, w_r)
    ids, w, _ = oracle.topk_gating(s, 2, oracle.GATE_TOPK_SOFTMAX)
    d = float(np.float32(0.41)) - float(np.float32(0.36))
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-d)), abs=1e-15)
    assert w[0, 1] == pytest.approx(1.0 / (1.0 + math.exp(d)), abs=1e-15)
    assert w[0, 0] > 0.5 > w[0, 1]


def _random_logits(T, E, seed):
    return synth.normal((T, E), seed, 50, 1.5, torch.float32).numpy()


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (64, 8), (128, 8)])
def test_softmax_order_invariance(E, k):
    # Top-k-then-softmax and softmax-then-top-k keep the same experts (softmax
    # is monotone); the first sums to 1, the second to less than 1, and
    # renormalising the second gives the first.
    s = _random_logits(2500, E, seed=E + k)
    ids_a, w_a, _ = oracle.topk_gating(s, k, oracle.GATE_TOPK_SOFTMAX)
    ids_b, w_b, _ = oracle.topk_gating(s, k, oracle.GATE_SOFTMAX_TOPK)
    ids_c, w_c, _ = oracle.topk_gating(s, k, oracle.GATE_SOFTMAX_TOPK_RENORM)
    assert np.array_equal(ids_a, ids_b) and np.array_equal(ids_a, ids_c)
    assert np.allclose(w_a.sum(1), 1.0, atol=1e-12, rtol=0)
    assert np.all(w_b.sum(1) < 1.0)
    assert np.allclose(w_c, w_a, atol=1e-12, rtol=0)
    # selected = the k largest logits (numpy argsort as the library routine)
    order = np.argsort(-s.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids_a, order)
    # weights are decreasing along the slots
    assert np.all(np.diff(w_a, axis=1) <= 0)


def test_softmax_topk_unnormalised_equals_full_softmax_entries():
    s = _random_logits(300, 32, seed=7)
    ids, w, _ = oracle.topk_gating(s, 4, oracle.GATE_SOFTMAX_TOPK)
    full = torch.softmax(torch.from_numpy(s).double(), dim=1).numpy()   # library softmax
    assert np.allclose(w, np.take_along_axis(full, ids.astype(np.int64), 1), atol=1e-14, rtol=0)


def test_sigmoid_variant_bias_selects_but_does_not_weight():
    T, E, k = 400, 64, 8
    s = _random_logits(T, E, seed=11)
    zero = np.zeros(E, dtype=np.float32)
    ids0, w0, _ = oracle.topk_gating(s, k, oracle.GATE_SIGMOID_BIAS_RENORM, zero)
    # b = 0: sigmoid is monotone, so the selection is the top-k of the logits
    ids_ref, _, _ = oracle.topk_gating(s, k, oracle.GATE_TOPK_SOFTMAX)
    assert np.array_equal(ids0, ids_ref)
    assert np.allclose(w0.sum(1), 1.0, atol=1e-12, rtol=0)
    # weight ratios are ratios of sigmoid affinities (torch.sigmoid as library)
    sig = torch.sigmoid(torch.from_numpy(s).double()).numpy()
    a = np.take_along_axis(sig, ids0.astype(np.int64), 1)
    assert np.allclose(w0 / w0[:, :1], a / a[:, :1], atol=1e-12, rtol=0)
    # a large bias on one expert forces it into every selection ...
    hot = 17
    big = zero.copy()
    big[hot] = 10.0
    ids1, w1, _ = oracle.topk_gating(s, k, oracle.GATE_SIGMOID_BIAS_RENORM, big)
    assert np.all((ids1 == hot).sum(1) == 1)
    # ... yet its weight is its own affinity over the selected affinities
    for t in range(T):
        sel = ids1[t]
        j = int(np.where(sel == hot)[0][0])
        assert w1[t, j] == pytest.approx(sig[t, hot] / sig[t, sel].sum(), abs=1e-12)
    # a bias that does not change the selection does not change the weights
    tiny = np.full(E, 1e-3, dtype=np.float32)
    ids2, w2, _ = oracle.topk_gating(s, k, oracle.GATE_SIGMOID_BIAS_RENORM, tiny)
    same = np.all(ids2 == ids0, axis=1)
    assert same.sum() > T // 2
    assert np.array_equal(w2[same], w0[same])


@pytest.mark.parametrize("mode", MODES)
def test_ties_go_to_lower_index(mode):
    E, k = 16, 5
    s = np.zeros((3, E), dtype=np.float32)
    s[1, [3, 9, 12]] = 0.25           # three equal maxima, then a 13-way tie
    s[2] = 1.0
    ids, w, gap = oracle.topk_gating(s, k, mode, np.zeros(E, dtype=np.float32))
    assert ids[0].tolist() == [0, 1, 2, 3, 4]
    assert ids[1].tolist() == [3, 9, 12, 0, 1]
    assert ids[2].tolist() == [0, 1, 2, 3, 4]
    assert gap[0] == 0.0 and gap[2] == 0.0


def test_gap_and_k_equals_E():
    s = _random_logits(50, 8, seed=5)
    ids, w, gap = oracle.topk_gating(s, 3, oracle.GATE_TOPK_SOFTMAX)
    srt = -np.sort(-s, axis=1)
    assert np.allclose(gap, srt[:, 2].astype(np.float64) - srt[:, 3], atol=0, rtol=0)
    ids, w, gap = oracle.topk_gating(s, 8, oracle.GATE_TOPK_SOFTMAX)
    assert np.all(np.isnan(gap))
    assert np.array_equal(np.sort(ids, 1), np.tile(np.arange(8), (50, 1)))


# ---------------------------------------------------------------- dispatch --

def test_dispatch_page_example():
    kv, _ = golden("dispatch_5token.txt")
    E, k = int(kv["E"][0]), int(kv["k"][0])
    ids = np.array([int(v) for v in kv["ids"]], dtype=np.int32).reshape(-1, k)
    counts, offsets, perm_src, inv_pos = oracle.dispatch(ids, E)
    assert counts.tolist() == [int(v) for v in kv["counts"]]
    assert offsets.tolist() == [0] + list(itertools.accumulate(int(v) for v in kv["counts"]))
    segs = " ".join(kv["segments"]).split("|")
    expect = [int(v) for seg in segs for v in seg.split()]
    assert perm_src.tolist() == expect                  # [t3][t1][t0,t2][t4]
    assert inv_pos.tolist() == [2, 1, 3, 0, 4]
    assert oracle.imbalance(counts, ids.size) == (16, 5)  # 2 / (5/8) = 3.2


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (7, 3, 5, 1), (1000, 8, 64, 2), (333, 2, 8, 3),
                                        (64, 8, 256, 4)])
def test_dispatch_invariants_and_sort(T, k, E, seed):
    ids = synth.random_ids(T, k, E, seed).numpy()
    counts, offsets, perm_src, inv_pos = oracle.dispatch(ids, E)
    flat = ids.reshape(-1)
    Na = T * k
    assert counts.sum() == Na and offsets[0] == 0 and offsets[-1] == Na
    assert np.array_equal(np.bincount(flat, minlength=E), counts)       # library histogram
    assert np.array_equal(np.concatenate([[0], np.cumsum(counts)]), offsets)
    assert np.array_equal(inv_pos[perm_src], np.arange(Na))
    assert np.array_equal(perm_src[inv_pos], np.arange(Na))
    # stable sort by (expert, token) as the independent formulation
    ref = sorted(range(Na), key=lambda a: (flat[a], a))
    assert perm_src.tolist() == ref
    for e in range(E):
        seg = perm_src[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // k) > 0)     # ascending token order
    num, den = oracle.imbalance(counts, Na)
    assert Fraction(num, den) == Fraction(int(counts.max()) * E, Na)


def test_dispatch_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0], [8]], dtype=np.int32), 8)
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0], [-1]], dtype=np.int32), 8)


# ----------------------------------------------------------- expert FFN --

def _dense_swiglu_torch(x, w13, w2):
    """Library reference: W2 @ (silu(W_gate x) * (W_up x)) in float64, with
    torch's matmul and silu."""
    I = w13.shape[0] // 2
    xd, gd, dd = x.double(), w13.double(), w2.double()
    return dd @ (torch.nn.functional.silu(gd[:I] @ xd) * (gd[I:] @ xd))


def _tiny_layer(T, H, I, E, seed, shared=False):
    x = synth.normal((T, H), seed, 1, 1.0, torch.bfloat16)
    w13 = synth.normal((E, 2 * I, H), seed, 4, H ** -0.5, torch.bfloat16)
    w2 = synth.normal((E, H, I), seed, 5, I ** -0.5, torch.bfloat16)
    w13s = w2s = None
    if shared:
        w13s = synth.normal((2 * I, H), seed, 6, H ** -0.5, torch.bfloat16)
        w2s = synth.normal((H, I), seed, 7, I ** -0.5, torch.bfloat16)
    return x, w13, w2, w13s, w2s


def test_expert_ffn_matches_library_swiglu():
    x, w13, w2, _, _ = _tiny_layer(3, 64, 32, 2, seed=1)
    for t in range(3):
        for e in range(2):
            got = oracle.expert_ffn(x[t], w13[e], w2[e])
            ref = _dense_swiglu_torch(x[t], w13[e], w2[e]).numpy()
            assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_gate_and_up_are_not_interchangeable():
    # With distinct gate and up blocks, swapping them changes the output, so
    # the pin above fixes which half of W13 is the gate.
    x, w13, w2, _, _ = _tiny_layer(1, 64, 32, 1, seed=2)
    swapped = torch.cat([w13[0, 32:], w13[0, :32]])
    a = oracle.expert_ffn(x[0], w13[0], w2[0])
    b = oracle.expert_ffn(x[0], swapped, w2[0])
    assert np.abs(a - b).max() > 1e-3


def test_k_equals_E_uniform_gates_is_dense_mean():
    # All logits 0 (W_r = 0) and k = E: top-k-then-softmax gives every expert
    # weight 1/E, so the layer is the mean of the E dense SwiGLU FFNs.
    T, H, I, E = 4, 64, 32, 4
    x, w13, w2, _, _ = _tiny_layer(T, H, I, E, seed=3)
    s = oracle.router_logits(x, torch.zeros((E, H)))
    assert np.all(s == 0)
    ids, w, _ = oracle.topk_gating(s, E, oracle.GATE_TOPK_SOFTMAX)
    assert np.allclose(w, 1.0 / E, atol=1e-15, rtol=0)
    y = oracle.layer_tokens(x, ids, w, w13, w2, range(T))
    for t in range(T):
        ref = sum(_dense_swiglu_torch(x[t], w13[e], w2[e]) for e in range(E)) / E
        assert np.allclose(y[t], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_single_expert_with_shared_expert():
    # E = 1, k = 1: the routed part is one plain SwiGLU FFN with weight 1, and
    # the shared expert adds its own FFN with weight 1.
    T, H, I = 3, 64, 32
    x, w13, w2, w13s, w2s = _tiny_layer(T, H, I, 1, seed=4, shared=True)
    s = oracle.router_logits(x, torch.zeros((1, H)))
    ids, w, _ = oracle.topk_gating(s, 1, oracle.GATE_SIGMOID_BIAS_RENORM, np.zeros(1, np.float32))
    assert np.array_equal(w, np.ones((T, 1)))
    y_routed = oracle.layer_tokens(x, ids, w, w13, w2, range(T))
    y_all = oracle.layer_tokens(x, ids, w, w13, w2, range(T), w13s, w2s)
    for t in range(T):
        r = _dense_swiglu_torch(x[t], w13[0], w2[0])
        sh = _dense_swiglu_torch(x[t], w13s, w2s)
        assert np.allclose(y_routed[t], r.numpy(), rtol=1e-12, atol=1e-13)
        assert np.allclose(y_all[t], (r + sh).numpy(), rtol=1e-12, atol=1e-13)


def test_weighted_combine_brute_force():
    # y_t = sum_j w_tj FFN_{id_tj}(x_t) with arbitrary ids / weights.
    T, H, I, E, k = 5, 64, 32, 6, 3
    x, w13, w2, _, _ = _tiny_layer(T, H, I, E, seed=5)
    ids = synth.random_ids(T, k, E, seed=5).numpy()
    w = np.abs(synth.normal((T, k), 5, 60, 1.0, torch.float64).numpy())
    y = oracle.layer_tokens(x, ids, w, w13, w2, range(T))
    for t in range(T):
        ref = sum(w[t, j] * _dense_swiglu_torch(x[t], w13[ids[t, j]], w2[ids[t, j]]) for j in range(k))
        assert np.allclose(y[t], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_dropless_batch_independence():
    # A token's output does not depend on the rest of its batch.
    inp = synth.make_layer(synth.CONFIGS["tiny"], 16, seed=6)
    y_batch, r = oracle.layer(inp)
    for t in (0, 7, 15):
        one = synth.LayerInputs(inp.cfg, 1, inp.seed, inp.x[t:t + 1].clone(), inp.w_router, None,
                                inp.w13, inp.w2)
        y1, r1 = oracle.layer(one)
        assert np.array_equal(r1["ids"][0], r["ids"][t])
        assert np.array_equal(y1[0], y_batch[t])


def test_layer_sample_rows_equal_full_batch_rows():
    inp = synth.make_layer(synth.CONFIGS["tiny"], 32, seed=8)
    y_all, _ = oracle.layer(inp)
    y_some, _ = oracle.layer(inp, tokens=[31, 2, 17])
    assert np.array_equal(y_some, y_all[[31, 2, 17]])
