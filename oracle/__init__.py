"""Python wrapper of the C oracle (``oracle/moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the plain fp64 CPU definition of the MoE FFN layer
forward that the CUDA library is checked against.  Only the test suite, the
smoke check and the benchmark's CPU-baseline leg use it; the product path never
imports it.  It shares no code with the CUDA library.

Inputs are torch CPU tensors (bf16 / fp32 / int32) or numpy arrays; outputs are
numpy arrays.  The shared library is compiled on first use (``build()``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

GATE_TOPK_SOFTMAX = 0
GATE_SOFTMAX_TOPK = 1
GATE_SOFTMAX_TOPK_RENORM = 2
GATE_SIGMOID_BIAS_RENORM = 3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (gcc, OpenMP).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle gives the same bits on x86-64 and aarch64."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_router_logits.argtypes = [P, P, I64, I64, I64, P, I32]
        lib.oracle_router_logits.restype = None
        lib.oracle_topk_gating.argtypes = [P, P, I64, I64, I64, I32, P, P, P]
        lib.oracle_topk_gating.restype = I32
        lib.oracle_dispatch.argtypes = [P, I64, I64, I64, P, P, P, P]
        lib.oracle_dispatch.restype = I32
        lib.oracle_imbalance.argtypes = [P, I64, I64, P, P]
        lib.oracle_imbalance.restype = None
        lib.oracle_expert_ffn.argtypes = [P, P, P, I64, I64, P]
        lib.oracle_expert_ffn.restype = None
        lib.oracle_layer_tokens.argtypes = [P, I64, I64, I64, P, P, P, P, P, P, P, I64, P, I32]
        lib.oracle_layer_tokens.restype = None
        lib.oracle_quantize_fp8.argtypes = [P, I64, I64, I64, P, P, I32]
        lib.oracle_quantize_fp8.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I32
        _lib = lib
    return _lib


def _u16(t) -> np.ndarray:
    """bf16 torch tensor (or uint16/int16 numpy array) -> contiguous uint16 array."""
    if isinstance(t, torch.Tensor):
        assert t.dtype == torch.bfloat16, t.dtype
        return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.asarray(t)
    assert a.dtype in (np.uint16, np.int16)
    return np.ascontiguousarray(a.view(np.uint16))


def _np(t, dtype) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=dtype))


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def router_logits(x, w_router, nthreads: int = 0) -> np.ndarray:
    """float32 logits s[T,E] (exact double dot product rounded once)."""
    xa = _u16(x)
    wr = _np(w_router, np.float32)
    T, H = xa.shape
    E = wr.shape[0]
    assert wr.shape[1] == H
    s = np.empty((T, E), dtype=np.float32)
    _load().oracle_router_logits(_p(xa), _p(wr), T, H, E, _p(s), nthreads or max_threads())
    return s


def topk_gating(s, k: int, mode: int, sel_bias=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(ids[T,k] int32, w[T,k] float64, gap[T] float64) from float32 logits."""
    sa = _np(s, np.float32)
    T, E = sa.shape
    b = None if sel_bias is None else _np(sel_bias, np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    gap = np.empty((T,), dtype=np.float64)
    rc = _load().oracle_topk_gating(_p(sa), None if b is None else _p(b), T, E, k, mode,
                                     _p(ids), _p(w), _p(gap))
    if rc != 0:
        raise ValueError("oracle_topk_gating: bad arguments")
    return ids, w, gap


def dispatch(ids, E: int):
    """(counts[E], offsets[E+1], perm_src[T*k], inv_pos[T*k]) int32."""
    ia = _np(ids, np.int32)
    T, k = ia.shape if ia.ndim == 2 else (ia.shape[0], 1)
    counts = np.empty((E,), dtype=np.int32)
    offsets = np.empty((E + 1,), dtype=np.int32)
    perm_src = np.empty((T * k,), dtype=np.int32)
    inv_pos = np.empty((T * k,), dtype=np.int32)
    rc = _load().oracle_dispatch(_p(ia), T, k, E, _p(counts), _p(offsets), _p(perm_src), _p(inv_pos))
    if rc != 0:
        raise ValueError("oracle_dispatch: expert id out of range")
    return counts, offsets, perm_src, inv_pos


# ---------------------------------------------- capacity and token dropping --
# "MoE推理优化全景指南", section "Capacity、padding 与 token dropping": an expert's
# capacity is C = ceil(capacity_factor * N_a / E); assignments beyond C are
# dropped.  CS349D lecture 8 notes, section 1.4 ("容量因子与丢 token"): a dropped
# (token, expert) pair contributes 0, nothing else changes.  Reading: the
# first C assignments of each expert in token order are kept (the dispatch
# layout's order inside a segment); the kept gate weights are not
# renormalised.

def expert_capacity(cf_num: int, cf_den: int, n_assign: int, E: int) -> int:
    """C = ceil(cf * N_a / E) for a capacity factor cf = cf_num / cf_den, in
    exact integer arithmetic."""
    if cf_num <= 0 or cf_den <= 0 or E <= 0 or n_assign <= 0:
        raise ValueError("capacity factor, assignments and experts must be positive")
    num, den = cf_num * n_assign, cf_den * E
    return -(-num // den)


def capacity_dispatch(ids, E: int, C: int):
    """The dispatch of the kept assignments: (counts[E] kept per expert,
    offsets[E+1], perm_src[n_kept] position -> assignment, inv_pos[T*k]
    assignment -> position or -1 when dropped).  Kept: the first C
    assignments of each expert in token order."""
    counts, offsets, perm, _ = dispatch(ids, E)
    n = perm.shape[0]
    kept = np.minimum(counts, C).astype(np.int32)
    offs = np.zeros(E + 1, dtype=np.int32)
    perm_c = []
    inv_c = np.full(n, -1, dtype=np.int32)
    for e in range(E):
        offs[e] = len(perm_c)
        for r in range(int(kept[e])):
            a = int(perm[offsets[e] + r])
            inv_c[a] = len(perm_c)
            perm_c.append(a)
    offs[E] = len(perm_c)
    return kept, offs, np.asarray(perm_c, dtype=np.int32), inv_c


def kept_weights(ids, w, E: int, C: int) -> np.ndarray:
    """Gate weights with every dropped assignment's weight set to 0 (its
    contribution to the layer output); the kept weights unchanged."""
    ia = _np(ids, np.int32)
    _, _, _, inv_c = capacity_dispatch(ia, E, C)
    wk = np.array(_np(w, np.float64), copy=True).reshape(-1)
    wk[inv_c < 0] = 0.0
    return wk.reshape(ia.shape)


# --------------------------------------------------- FP8 expert weights --
# "MoE推理优化全景指南", section "量化与 offload 并非独立开关", "专家权重量化":
# FP8 expert weights cut weight capacity and bandwidth; the scale layout is
# the implementation's choice.  Reading: OCP FP8 E4M3 ("fn": no infinities;
# 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; normal values
# 2^(E-7) * (1 + m/8), subnormal m * 2^-9, largest 448, code 0x7F / 0xFF is
# NaN), one power-of-two scale 2^s per block of 128 rows x 128 columns of each
# weight matrix, s the smallest integer with max|w| / 2^s <= 448, codes by
# round-to-nearest-even of w / 2^s, saturating at +-448.  A power-of-two scale
# makes code * 2^s exact in bf16, so the dequantised weights are bf16 tensors
# and the layer is the unchanged definition over them.

FP8_BLOCK = 128
FP8_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of E4M3 codes (uint8 array); NaN for 0x7F / 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m.astype(np.float64), -9)
    v = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest value, ties to the even code
    (mantissa bit 0 clear), saturating at +-448; the sign bit follows the
    value's sign (so -0 gives 0x80).  Below 2^-6 the codes are multiples of
    2^-9 (code = m); in the binade [2^e, 2^(e+1)) they are 2^e * (1 + m/8)
    (code = (e + 7) * 8 + m), and rounding m up to 8 is the next binade's
    first code."""
    a = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(a), FP8_MAX)
    sub = mag < 2.0 ** -6
    _, x = np.frexp(np.where(sub, 1.0, mag))      # mag = f * 2^x, f in [0.5, 1)
    e = x.astype(np.int64) - 1                     # mag in [2^e, 2^(e+1))
    m_norm = np.rint((np.ldexp(np.where(sub, 1.0, mag), -e) - 1.0) * 8.0).astype(np.int64)
    code_norm = (e + 7) * 8 + m_norm
    code_sub = np.rint(np.ldexp(mag, 9)).astype(np.int64)   # 0 .. 8 (8 = 2^-6, code 0x08)
    code = np.minimum(np.where(sub, code_sub, code_norm), 0x7E)
    code = code | np.where(np.signbit(a), 0x80, 0)
    return code.astype(np.uint8)


def fp8_block_exponent(amax: float) -> int:
    """The smallest integer s with amax / 2^s <= 448 (0 for an all-zero
    block), clamped to [-15, 7]."""
    return int(_block_exponents(np.asarray([amax], dtype=np.float64))[0])


FP8_EXP_MIN, FP8_EXP_MAX = -15, 7   # code * 2^s exact in fp16 (and bf16)


def _block_exponents(amax: np.ndarray) -> np.ndarray:
    _, x = np.frexp(amax)
    s = x.astype(np.int64) - 9                     # amax / 2^s in [256, 512)
    s = np.where(np.ldexp(amax, -s) > FP8_MAX, s + 1, s)
    s = np.where(np.ldexp(amax, -(s - 1)) <= FP8_MAX, s - 1, s)
    s = np.clip(s, FP8_EXP_MIN, FP8_EXP_MAX)
    return np.where(amax == 0.0, 0, s)


def quantize_fp8(w) -> Tuple[np.ndarray, np.ndarray]:
    """E4M3 codes [n, rows, K] and block exponents [n, ceil(rows/128),
    ceil(K/128)] (int8) of bf16 matrices w [n, rows, K]: per 128 x 128
    block, s = the smallest integer with max|w| / 2^s <= 448, then the codes
    of w / 2^s."""
    wa = w.double().numpy() if isinstance(w, torch.Tensor) else _np(w, np.float64)
    n, rows, K = wa.shape
    B = FP8_BLOCK
    nr, nk = -(-rows // B), -(-K // B)
    pad = np.zeros((n, nr * B, nk * B))
    pad[:, :rows, :K] = wa
    blocks = pad.reshape(n, nr, B, nk, B)
    amax = np.max(np.abs(blocks), axis=(2, 4))                       # [n, nr, nk]
    sc = _block_exponents(amax)
    scaled = np.ldexp(blocks, -sc[:, :, None, :, None])
    q = e4m3_encode(scaled).reshape(n, nr * B, nk * B)[:, :rows, :K]
    return np.ascontiguousarray(q), sc.astype(np.int8)


def quantize_fp8_c(w, nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """quantize_fp8 by the oracle's C implementation (the same definition,
    block by block, OpenMP over blocks): for large weight sets."""
    wa = _u16(w)
    n, rows, K = wa.shape
    nr, nk = -(-rows // FP8_BLOCK), -(-K // FP8_BLOCK)
    q = np.empty((n, rows, K), dtype=np.uint8)
    sc = np.empty((n, nr, nk), dtype=np.int8)
    _load().oracle_quantize_fp8(_p(wa), n, rows, K, _p(q), _p(sc), nthreads or max_threads())
    return q, sc


def dequantize_fp8(q, sc) -> torch.Tensor:
    """bf16 tensor [n, rows, K] of code * 2^s (exact in bf16)."""
    qa = np.asarray(q, dtype=np.uint8)
    n, rows, K = qa.shape
    B = FP8_BLOCK
    s = np.asarray(sc, dtype=np.int64)
    full = np.repeat(np.repeat(s, B, axis=1), B, axis=2)[:, :rows, :K]
    v = np.ldexp(e4m3_decode(qa), full)
    t = torch.from_numpy(v).to(torch.bfloat16)
    if not np.array_equal(t.double().numpy(), v):
        raise ValueError("dequantised weights not exact in bf16")
    return t


def imbalance(counts, n_assign: int) -> Tuple[int, int]:
    """Imbalance ratio max_e n_e / (N_a/E) as an exact fraction (num, den)."""
    c = _np(counts, np.int32)
    num = ctypes.c_int64()
    den = ctypes.c_int64()
    _load().oracle_imbalance(_p(c), c.shape[0], n_assign, ctypes.byref(num), ctypes.byref(den))
    return int(num.value), int(den.value)


def expert_ffn(x_row, w13_e, w2_e) -> np.ndarray:
    xa, g, d = _u16(x_row), _u16(w13_e), _u16(w2_e)
    H = xa.shape[-1]
    I = g.shape[0] // 2
    out = np.empty((H,), dtype=np.float64)
    _load().oracle_expert_ffn(_p(xa), _p(g), _p(d), H, I, _p(out))
    return out


def layer_tokens(x, ids, w, w13, w2, tokens: Sequence[int], w13_shared=None, w2_shared=None,
                 nthreads: int = 0) -> np.ndarray:
    """y[n,H] (float64) for token indices ``tokens``.

    ``w13``/``w2`` are [E,2I,H]/[E,H,I] bf16 tensors or dicts {expert: block}
    holding at least the experts the listed tokens select."""
    xa = _u16(x)
    T, H = xa.shape
    ia = _np(ids, np.int32)
    wa = _np(w, np.float64)
    k = ia.shape[1]
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    need = sorted({int(e) for e in ia[toks].reshape(-1)}) if len(toks) else []
    if isinstance(w13, dict):
        E = max(max(w13.keys()) + 1, int(ia.max()) + 1)
        blocks13 = {e: _u16(w13[e]) for e in need}
        blocks2 = {e: _u16(w2[e]) for e in need}
    else:
        E = w13.shape[0]
        blocks13 = {e: _u16(w13[e]) for e in need}
        blocks2 = {e: _u16(w2[e]) for e in need}
    some = next(iter(blocks13.values())) if blocks13 else None
    I = (some.shape[0] // 2) if some is not None else (_u16(w13_shared).shape[0] // 2)
    p13 = (ctypes.c_void_p * E)()
    p2 = (ctypes.c_void_p * E)()
    for e in need:
        p13[e] = _p(blocks13[e])
        p2[e] = _p(blocks2[e])
    s13 = None if w13_shared is None else _u16(w13_shared)
    s2 = None if w2_shared is None else _u16(w2_shared)
    y = np.empty((len(toks), H), dtype=np.float64)
    _load().oracle_layer_tokens(_p(xa), H, I, k, _p(ia), _p(wa), p13, p2,
                                None if s13 is None else _p(s13), None if s2 is None else _p(s2),
                                _p(toks), len(toks), _p(y), nthreads or max_threads())
    return y


def route(inputs, nthreads: int = 0) -> Dict[str, np.ndarray]:
    """Router + gating of a ``synth.LayerInputs`` batch: logits, ids, w, gap."""
    s = router_logits(inputs.x, inputs.w_router, nthreads)
    ids, w, gap = topk_gating(s, inputs.cfg.k, inputs.cfg.gating, inputs.sel_bias)
    return {"logits": s, "ids": ids, "w": w, "gap": gap}


def layer(inputs, tokens: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Full layer forward of a ``synth.LayerInputs`` batch (optionally only some
    tokens' outputs).  Returns (y[n,H] float64, routing dict)."""
    r = route(inputs, nthreads)
    if tokens is None:
        tokens = range(inputs.T)
    y = layer_tokens(inputs.x, r["ids"], r["w"], inputs.w13, inputs.w2, list(tokens),
                     inputs.w13_shared, inputs.w2_shared, nthreads)
    return y, r


# ------------------------------------------------- EP <-> TP weight reshard --
# Moebius, section 3.1 "Weights Resharding" and Figure 4.  Under expert
# parallelism a rank holds E_l complete experts, W13 [E_l, 2I, H] (gate rows
# [0,I), up rows [I,2I)) and W2 [E_l, H, I]; under tensor parallelism each of P
# ranks holds slice p of the intermediate dimension of every expert.  The
# EP -> TP local permute packs one chunk per peer: chunk p of expert e is
# W13 rows (gate slice p, then up slice p) and W2 columns slice p.  Written as
# the index permutation itself (reshape + transpose; no arithmetic), on any
# element type.

def reshard_pack(w13, w2, P: int):
    """EP -> TP: (w13 [E_l,2I,H], w2 [E_l,H,I]) -> (w13_chunks [P,E_l,2I/P,H],
    w2_chunks [P,E_l,H,I/P]); either may be None."""
    c13 = c2 = None
    if w13 is not None:
        a = np.asarray(w13)
        E_l, two_i, H = a.shape
        Ip = two_i // 2 // P
        # [e][g][p][r][h] -> [p][e][g][r][h]
        c13 = np.ascontiguousarray(
            a.reshape(E_l, 2, P, Ip, H).transpose(2, 0, 1, 3, 4).reshape(P, E_l, 2 * Ip, H))
    if w2 is not None:
        a = np.asarray(w2)
        E_l, H, I = a.shape
        # [e][h][p][c] -> [p][e][h][c]
        c2 = np.ascontiguousarray(a.reshape(E_l, H, P, I // P).transpose(2, 0, 1, 3))
    return c13, c2


def reshard_unpack(w13_chunks, w2_chunks, P: int):
    """TP -> EP: the inverse of reshard_pack (chunk index = source peer)."""
    w13 = w2 = None
    if w13_chunks is not None:
        a = np.asarray(w13_chunks)
        _, E_l, two_ip, H = a.shape
        Ip = two_ip // 2
        # [p][e][g][r][h] -> [e][g][p][r][h]
        w13 = np.ascontiguousarray(
            a.reshape(P, E_l, 2, Ip, H).transpose(1, 2, 0, 3, 4).reshape(E_l, 2 * P * Ip, H))
    if w2_chunks is not None:
        a = np.asarray(w2_chunks)
        _, E_l, H, Ip = a.shape
        # [p][e][h][c] -> [e][h][p][c]
        w2 = np.ascontiguousarray(a.transpose(1, 2, 0, 3).reshape(E_l, H, P * Ip))
    return w13, w2
