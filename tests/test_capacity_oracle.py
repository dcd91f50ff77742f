"""Pins of the oracle's capacity-factor dispatch ("MoE推理优化全景指南",
"Capacity、padding 与 token dropping": C = ceil(capacity factor x N_a / E),
assignments beyond C dropped; CS349D lecture 8 notes, section 1.4: a dropped
pair contributes 0, and with a capacity limit a token's output depends on the
rest of its batch)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden


def test_capacity_formula_examples():
    # the page's formula in exact arithmetic
    assert oracle.expert_capacity(5, 4, 5, 8) == 1          # 1.25 * 5 / 8 = 0.78125
    assert oracle.expert_capacity(1, 1, 16, 8) == 2         # exactly 2
    assert oracle.expert_capacity(1, 1, 17, 8) == 3         # 2.125
    assert oracle.expert_capacity(2, 1, 8192 * 8, 128) == 1024
    assert oracle.expert_capacity(5, 4, 1024 * 8, 128) == 80
    with pytest.raises(ValueError):
        oracle.expert_capacity(0, 1, 5, 8)


def test_capacity_page_example():
    kv, _ = golden("dispatch_5token.txt")
    ids = np.array([int(v) for v in kv["ids"]], dtype=np.int32).reshape(-1, 1)
    E = int(kv["E"][0])
    num, den = (int(v) for v in kv["capacity_factor"])
    C = oracle.expert_capacity(num, den, ids.size, E)
    assert C == int(kv["capacity"][0])
    counts, offsets, perm, inv = oracle.capacity_dispatch(ids, E, C)
    segs = " ".join(kv["kept_segments"]).split("|")
    want = [int(t) for seg in segs for t in seg.split()]
    assert perm.tolist() == want
    assert counts.tolist() == [1, 1, 0, 1, 0, 0, 1, 0]
    assert offsets.tolist() == [0, 1, 2, 2, 3, 3, 3, 4, 4]
    dropped = [int(v) for v in kv["dropped"]]
    assert [a for a in range(ids.size) if inv[a] < 0] == dropped


@pytest.mark.parametrize("T,k,E,seed", [(64, 2, 8, 1), (300, 8, 32, 2), (50, 4, 4, 3)])
def test_large_capacity_is_dropless(T, k, E, seed):
    ids = synth.random_ids(T, k, E, seed).numpy()
    c, o, p, i = oracle.dispatch(ids, E)
    kc, ko, kp, ki = oracle.capacity_dispatch(ids, E, int(c.max()))
    assert np.array_equal(kc, c) and np.array_equal(ko, o)
    assert np.array_equal(kp, p) and np.array_equal(ki, i)


@pytest.mark.parametrize("C", [1, 3, 10])
def test_kept_are_first_in_token_order_brute_force(C):
    T, k, E = 80, 4, 8
    ids = synth.skewed_ids(T, k, E, 7, hot=2).numpy()
    counts, offsets, perm, inv = oracle.capacity_dispatch(ids, E, C)
    seen = np.zeros(E, dtype=np.int64)
    for t in range(T):                        # walk the batch in token order
        for j in range(k):
            a, e = t * k + j, int(ids[t, j])
            if seen[e] < C:
                assert inv[a] >= 0 and perm[inv[a]] == a
                assert offsets[e] <= inv[a] < offsets[e + 1]
            else:
                assert inv[a] == -1
            seen[e] += 1
    assert np.array_equal(counts, np.minimum(seen, C))
    assert counts.sum() == perm.size <= min(T * k, E * C)
    # positions inside a segment ascend with the token
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_dropped_pairs_contribute_zero_and_make_outputs_batch_dependent():
    # token 2 picks expert 0 in both batches; with capacity 2 it is dropped
    # where two earlier tokens also picked expert 0 and kept where none did:
    # its output depends on its neighbours (dropless: the same in both)
    H, I, E, k = 64, 64, 2, 1
    w13 = synth.normal((E, 2 * I, H), 1, 4, H ** -0.5, torch.bfloat16)
    w2 = synth.normal((E, H, I), 1, 5, I ** -0.5, torch.bfloat16)
    x = synth.normal((4, H), 1, 1, 1.0, torch.bfloat16)
    w = np.ones((4, k))
    C = 2
    crowded = np.array([[0], [0], [0], [1]], dtype=np.int32)   # token 2 is expert 0's third
    alone = np.array([[1], [1], [0], [1]], dtype=np.int32)     # token 2 is expert 0's first
    y_c = oracle.layer_tokens(x, crowded, oracle.kept_weights(crowded, w, E, C), w13, w2, [2])
    y_a = oracle.layer_tokens(x, alone, oracle.kept_weights(alone, w, E, C), w13, w2, [2])
    assert np.all(y_c == 0.0)                 # dropped: contributes 0
    assert np.max(np.abs(y_a)) > 0            # kept in the other batch
    # dropless: the token's output is the same in both batches
    y_c0 = oracle.layer_tokens(x, crowded, w, w13, w2, [2])
    y_a0 = oracle.layer_tokens(x, alone, w, w13, w2, [2])
    assert np.array_equal(y_c0, y_a0)
    # kept weights are not renormalised
    wk = oracle.kept_weights(crowded, w, E, C)
    assert wk[:, 0].tolist() == [1.0, 1.0, 0.0, 1.0]
