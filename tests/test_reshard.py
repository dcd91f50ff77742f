"""EP <-> TP expert-weight reshard permute (Moebius, section 3.1 "Weights
Resharding" and Figure 4).

CPU: the oracle's permutation is pinned by a worked example written out by
hand from the definition, by the round trip, and by the meaning of the TP
layout -- the P shards of an expert, each run as a SwiGLU FFN of intermediate
size I/P, sum to the whole expert's FFN (a mismatched gate/up slice or a wrong
W2 column slice breaks it).  The C ABI rejects bad arguments before launching.

GPU: the CUDA permute is bit-exact against the oracle, at small ragged shapes
and at the Qwen3-235B per-rank shape (E_local = 16, P = 8)."""

import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_gb300 as moe


# ------------------------------------------------------------ oracle pins --

def test_pack_worked_example():
    # E_l = 2 experts, I = 4 (gate rows 0-3, up rows 4-7), H = 3, P = 2: slice
    # p of the intermediate dimension is gate rows {2p, 2p+1} and up rows
    # {4+2p, 5+2p}; W2 slice p is columns {2p, 2p+1}.
    w13 = np.arange(2 * 8 * 3).reshape(2, 8, 3)
    w2 = np.arange(2 * 3 * 4).reshape(2, 3, 4)
    c13, c2 = oracle.reshard_pack(w13, w2, 2)
    assert c13.shape == (2, 2, 4, 3) and c2.shape == (2, 2, 3, 2)
    # peer 0, expert 0: rows 0, 1 (gate) and 4, 5 (up) of expert 0
    assert c13[0, 0].tolist() == [[0, 1, 2], [3, 4, 5], [12, 13, 14], [15, 16, 17]]
    # peer 1, expert 1: rows 2, 3 and 6, 7 of expert 1 (values 24..47)
    assert c13[1, 1].tolist() == [[30, 31, 32], [33, 34, 35], [42, 43, 44], [45, 46, 47]]
    # peer 1, expert 0: columns 2, 3 of expert 0's W2
    assert c2[1, 0].tolist() == [[2, 3], [6, 7], [10, 11]]
    assert c2[0, 1].tolist() == [[12, 13], [16, 17], [20, 21]]


@pytest.mark.parametrize("E_l,H,I,P", [(1, 8, 8, 1), (3, 16, 48, 3), (2, 24, 64, 8)])
def test_unpack_inverts_pack(E_l, H, I, P):
    rng = np.random.default_rng(E_l * 100 + P)
    w13 = rng.integers(0, 1 << 16, size=(E_l, 2 * I, H), dtype=np.uint16)
    w2 = rng.integers(0, 1 << 16, size=(E_l, H, I), dtype=np.uint16)
    c13, c2 = oracle.reshard_pack(w13, w2, P)
    b13, b2 = oracle.reshard_unpack(c13, c2, P)
    assert np.array_equal(b13, w13) and np.array_equal(b2, w2)
    # a pure permutation: the same multiset of values
    assert np.array_equal(np.sort(c13.ravel()), np.sort(w13.ravel()))


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("P", [2, 4])
def test_tp_shards_sum_to_the_expert(P):
    """Tensor parallelism over the intermediate dimension: the P ranks' FFN
    outputs of one expert add up to the expert's output (fp64 oracle)."""
    rng = np.random.default_rng(7)
    E_l, H, I = 2, 64, 32
    w13 = _bf16(rng.normal(0, H ** -0.5, (E_l, 2 * I, H)))
    w2 = _bf16(rng.normal(0, I ** -0.5, (E_l, H, I)))
    x = _bf16(rng.normal(0, 1, (H,)))
    u13 = w13.view(torch.int16).numpy().view(np.uint16)
    u2 = w2.view(torch.int16).numpy().view(np.uint16)
    c13, c2 = oracle.reshard_pack(u13, u2, P)
    for e in range(E_l):
        full = oracle.expert_ffn(x, w13[e], w2[e])
        parts = sum(oracle.expert_ffn(x, c13[p, e], c2[p, e]) for p in range(P))
        assert np.allclose(parts, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
    # a shard whose up slice is taken from the neighbouring peer is not a TP shard
    bad = c13[0, 0].copy()
    bad[I // P:] = c13[1, 0][I // P:]
    wrong = oracle.expert_ffn(x, bad, c2[0, 0]) + sum(
        oracle.expert_ffn(x, c13[p, 0], c2[p, 0]) for p in range(1, P))
    assert not np.allclose(wrong, oracle.expert_ffn(x, w13[0], w2[0]), rtol=1e-6)


# ------------------------------------------------- host-side validation --

@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(moe.LIB_PATH):
        from routed_expert_ffn_gb300 import build
        build.build()
    return moe.library()


FAKE = [0x10000, 0x20000000, 0x40000000, 0x60000000]  # aligned, never dereferenced


@pytest.mark.parametrize("shape,code", [
    ((0, 64, 64, 2), moe.MOE_ERR_UNSUPPORTED_SHAPE),      # E_local < 1
    ((2, 60, 64, 2), moe.MOE_ERR_UNSUPPORTED_SHAPE),      # H % 8
    ((2, 64, 96, 5), moe.MOE_ERR_UNSUPPORTED_SHAPE),      # I % P
    ((2, 64, 36, 3), moe.MOE_ERR_UNSUPPORTED_SHAPE),      # (I/P) % 8
    ((512, 16384, 32768, 1), moe.MOE_ERR_UNSUPPORTED_SHAPE),  # >= 2^35 bytes
])
def test_reshard_rejects_bad_shapes(lib, shape, code):
    for fn in (lib.moe_reshard_ep_to_tp_pack, lib.moe_reshard_tp_to_ep_unpack):
        assert fn(*shape, *FAKE, None) == code


def test_reshard_rejects_bad_pointers(lib):
    a, b, c, d = FAKE
    f = lib.moe_reshard_ep_to_tp_pack
    assert f(2, 64, 64, 2, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert f(2, 64, 64, 2, a, None, c, d, None) == moe.MOE_ERR_INVALID_ARG   # w2 pair half-null
    assert f(2, 64, 64, 2, a + 8, b, c, d, None) == moe.MOE_ERR_INVALID_ARG  # misaligned
    assert f(2, 64, 64, 2, a, b, a + 1024, d, None) == moe.MOE_ERR_INVALID_ARG  # overlap


# ------------------------------------------------------------ GPU parity --

def _run(E_l, H, I, P, seed):
    g = torch.Generator().manual_seed(seed)
    w13 = torch.randint(-32768, 32767, (E_l, 2 * I, H), generator=g, dtype=torch.int16)
    w2 = torch.randint(-32768, 32767, (E_l, H, I), generator=g, dtype=torch.int16)
    want13, want2 = oracle.reshard_pack(w13.numpy(), w2.numpy(), P)
    d13, d2 = w13.cuda(), w2.cuda()
    c13 = torch.empty((P, E_l, 2 * I // P, H), dtype=torch.int16, device="cuda")
    c2 = torch.empty((P, E_l, H, I // P), dtype=torch.int16, device="cuda")
    moe.moe_reshard_ep_to_tp_pack(E_l, H, I, P, d13, d2, c13, c2)
    b13, b2 = torch.empty_like(d13), torch.empty_like(d2)
    moe.moe_reshard_tp_to_ep_unpack(E_l, H, I, P, c13, c2, b13, b2)
    torch.cuda.synchronize()
    assert np.array_equal(c13.cpu().numpy(), want13)
    assert np.array_equal(c2.cpu().numpy(), want2)
    # the unpack against the oracle's inverse of the oracle's chunks
    u13, u2 = oracle.reshard_unpack(want13, want2, P)
    assert np.array_equal(b13.cpu().numpy(), u13)
    assert np.array_equal(b2.cpu().numpy(), u2)


@pytest.mark.gpu
@pytest.mark.parametrize("E_l,H,I,P", [(1, 8, 8, 1), (3, 72, 96, 4), (5, 64, 256, 8),
                                       (2, 4096, 1536, 1)])
def test_gpu_reshard_small(E_l, H, I, P):
    _run(E_l, H, I, P, seed=E_l + P)


@pytest.mark.gpu
def test_gpu_reshard_qwen3_rank():
    # Qwen3-235B-A22B over 8 ranks: 16 experts per rank, I/P = 192
    _run(16, 4096, 1536, 8, seed=0)


@pytest.mark.gpu
def test_gpu_reshard_one_tensor_only():
    E_l, H, I, P = 2, 64, 128, 4
    w2 = torch.randint(-32768, 32767, (E_l, H, I), dtype=torch.int16)
    _, want2 = oracle.reshard_pack(None, w2.numpy(), P)
    c2 = torch.empty((P, E_l, H, I // P), dtype=torch.int16, device="cuda")
    moe.moe_reshard_ep_to_tp_pack(E_l, H, I, P, None, w2.cuda(), None, c2)
    torch.cuda.synchronize()
    assert np.array_equal(c2.cpu().numpy(), want2)
