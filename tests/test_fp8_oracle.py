"""Pins of the oracle's FP8 expert-weight format (E4M3 codes with a
power-of-two scale per 128 x 128 block; "MoE推理优化全景指南", "量化与 offload
并非独立开关", "专家权重量化": FP8 weights, with the scale layout the
implementation's choice).  The encoder is checked against torch's own
float8_e4m3fn conversion, the decoder against the format's definition
(specific codes and a full round trip), the block exponent against its
defining inequality, and the dequantised weights against bf16 exactness and
the rounding bound."""

import numpy as np
import pytest
import torch

import oracle
import synth


def test_e4m3_decode_known_codes():
    dec = oracle.e4m3_decode
    assert dec([0x00])[0] == 0.0
    assert dec([0x38])[0] == 1.0                 # E = 7, m = 0
    assert dec([0x7E])[0] == 448.0               # largest finite
    assert dec([0x01])[0] == 2.0 ** -9           # smallest subnormal
    assert dec([0x08])[0] == 2.0 ** -6           # smallest normal
    assert dec([0x07])[0] == 7 * 2.0 ** -9       # largest subnormal
    assert dec([0xB8])[0] == -1.0
    assert np.isnan(dec([0x7F])[0]) and np.isnan(dec([0xFF])[0])


def test_e4m3_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(v)
    # +0 and -0 both decode to 0.0; their sign is kept by the encoder
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch():
    # a dense grid over the finite range, every midpoint between neighbouring
    # codes (ties) and a jitter around them
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    grid = np.concatenate([np.linspace(0, 448, 20001), mids, mids * (1 + 1e-6),
                           mids * (1 - 1e-6), pos])
    grid = grid.astype(np.float32).astype(np.float64)   # values torch sees exactly
    grid = np.concatenate([grid, -grid])
    grid = grid[np.abs(grid) <= 448]
    ours = oracle.e4m3_encode(grid)
    ref = torch.from_numpy(grid.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # float32 cast of the grid first: compare on values exact in float32
    exact32 = grid.astype(np.float32).astype(np.float64) == grid
    assert np.array_equal(ours[exact32], ref[exact32])
    assert exact32.sum() > 20000


def test_e4m3_saturates():
    assert oracle.e4m3_encode([1e6])[0] == 0x7E
    assert oracle.e4m3_encode([-500.0])[0] == 0xFE


@pytest.mark.parametrize("amax", [1.0, 448.0, 448.0001, 0.0779, 0.01, 2.0 ** -14 * 448])
def test_block_exponent_is_the_smallest(amax):
    s = oracle.fp8_block_exponent(amax)
    assert amax / 2.0 ** s <= 448.0 < amax / 2.0 ** (s - 1)


def test_block_exponent_clamps_to_the_fp16_exact_range():
    assert oracle.fp8_block_exponent(3e-7) == -15          # would be -31
    assert oracle.fp8_block_exponent(2.0 ** -16 * 448) == -15
    assert oracle.fp8_block_exponent(1e6) == 7             # would be 12 (codes saturate)
    # every code times 2^s for s in [-15, 7] is exact in fp16
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    for s in (-15, -12, 0, 7):
        x = np.ldexp(v, s)
        assert np.array_equal(x.astype(np.float16).astype(np.float64), x)


def test_quantize_blocks_and_dequantise_exactly():
    w = synth.normal((3, 200, 300), 4, 9, 0.02, torch.bfloat16)
    w[1, 5:40, 10:90] *= 1000           # a block with a much larger range
    w[2, 128:, 256:] = 0                # an all-zero block (rows 128.., columns 256..)
    q, sc = oracle.quantize_fp8(w)
    assert q.shape == (3, 200, 300) and sc.shape == (3, 2, 3)
    assert sc[2, 1, 2] == 0 and np.all(q[2, 128:, 256:] == 0)
    deq = oracle.dequantize_fp8(q, sc)          # raises unless exact in bf16
    wd, dd = w.double().numpy(), deq.double().numpy()
    for i in range(3):
        for r in range(2):
            for c in range(3):
                blk = np.s_[i, r * 128:(r + 1) * 128, c * 128:(c + 1) * 128]
                s = int(sc[i, r, c])
                amax = np.max(np.abs(wd[blk]))
                assert amax / 2.0 ** s <= 448 or s == 7
                # rounding error: half a step of E4M3 at the value's binade
                # (2^-4 relative for normals), 2^-10 * 2^s absolute below
                err = np.abs(dd[blk] - wd[blk])
                bound = np.maximum(np.abs(wd[blk]) * 2.0 ** -4, 2.0 ** (s - 10))
                assert np.all(err <= bound)
    # the quantised layer's weights are within FP8 precision of the originals
    rel = np.linalg.norm(dd - wd) / np.linalg.norm(wd)
    assert rel < 0.03


def test_c_quantizer_equals_the_numpy_definition():
    w = synth.normal((4, 300, 448), 5, 3, 0.05, torch.bfloat16)
    w[0, :7, :] *= 3000                        # saturating-range block neighbours
    w[1, 128:256, 128:256] = 0
    w[2, 40, 17] = -0.0
    w[3] = (w[3].float() * 2.0 ** -30).to(torch.bfloat16)   # tiny values (negative exponents)
    qa, sa = oracle.quantize_fp8(w)
    qc, sc = oracle.quantize_fp8_c(w)
    assert np.array_equal(sa, sc)
    assert np.array_equal(qa, qc)
