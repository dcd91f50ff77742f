"""Seeded synthetic inputs for the MoE FFN layer forward.

This module is the one place both sides draw their inputs from: the CPU oracle
(test infrastructure) and the CUDA path.  It holds none of the layer's
arithmetic -- no routing, no gating, no expert FFN -- only a counter-based
random generator and the recipe that turns it into tensors of the workload
shapes.

Generator.  Element ``i`` of tensor ``tid`` under seed ``seed`` is a pure
function of ``(seed, tid, i)``:

* ``lowbias32`` integer hash (C. Wellons, "Prospecting for Hash Functions",
  2018: xorshift 16 / multiply 0x7feb352d / xorshift 15 / multiply 0x846ca68b /
  xorshift 16), evaluated with 64-bit integer tensor ops whose products never
  exceed 2**48, so the bits are identical on every device and host;
* two 32-bit words per element -> two uniforms -> one standard normal by the
  Box-Muller transform (G. Box and M. Muller, 1958), in float64;
* scaled by the requested standard deviation, rounded to float32, then (for
  bf16 tensors) rounded to bfloat16 with round-to-nearest-even.

Because every element is independent, a tensor can be produced in chunks, on
the GPU for the large weight sets, and any slice of it can be regenerated on
the host.  Parity tests never rely on that: they copy the exact bytes the GPU
consumed back to the host for the oracle.

Workload recipe (shapes from the five layer configurations):

* ``x[T,H]`` ~ N(0,1) as bf16.  When the configuration asks for a per-expert
  routing skew, channel 0 of every token is the constant 1.0 and the router
  column 0 carries the per-expert logit offset delta_e, so the plain linear
  router ``s = W_r x`` itself produces ``s_e + delta_e``;
* ``W_r[E,H]`` fp32 ~ N(0, 0.02^2);
* ``W13[E,2I,H]`` bf16 ~ N(0, 1/H) (rows ``[0,I)`` gate, ``[I,2I)`` up);
  ``W2[E,H,I]`` bf16 ~ N(0, 1/I); the shared expert likewise;
* selection-only bias ``b[E]`` ~ N(0, 0.1^2) for the sigmoid-gated layer;
* skew: ``delta_e ~ N(0, 0.5^2)`` (Mixtral-shaped layer) or a Zipf-shaped
  offset ``delta_e = -beta * s * ln(r_e)`` with ``r`` a seeded permutation of
  ``1..E`` (Qwen3 layers: s=1.1; DeepSeek-V3 layer: s=1.2, beta=1).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch

M32 = 0xFFFFFFFF

# Gating variant labels.  The numeric values are the C ABI's enum values.
GATE_TOPK_SOFTMAX = 0            # keep top-k logits, softmax over them (Mixtral)
GATE_SOFTMAX_TOPK = 1            # softmax over all experts, keep top-k, no renormalisation
GATE_SOFTMAX_TOPK_RENORM = 2     # as above, renormalised over the kept k (Qwen3)
GATE_SIGMOID_BIAS_RENORM = 3     # sigmoid affinity, selection-only bias, renormalised (DeepSeek-V3)

# Tensor ids: distinct streams of the counter generator.
TID_X, TID_WR, TID_BIAS, TID_W13, TID_W2, TID_W13S, TID_W2S, TID_PERM, TID_DELTA = range(1, 10)

# Zipf logit-offset scale for the Qwen3-shaped layers, chosen so that the
# realised imbalance ratio of the T=1024, seed-0 batch is close to 3 (the
# configuration's target).  tests/test_synth.py re-measures it with the oracle.
ZIPF_BETA_QWEN3 = 0.21


# ---------------------------------------------------------------- generator --

def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 x in [0, 2**32) without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _hash32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _hash32_int(v: int) -> int:
    v &= M32
    v ^= v >> 16
    v = (v * 0x7FEB352D) & M32
    v ^= v >> 15
    v = (v * 0x846CA68B) & M32
    v ^= v >> 16
    return v


def _keys(seed: int, tid: int) -> Tuple[int, int]:
    k1 = _hash32_int(_hash32_int(seed) ^ ((tid * 0x9E3779B9) & M32))
    k2 = _hash32_int(k1 ^ 0x85EBCA6B)
    return k1, k2


def _words(seed: int, tid: int, start: int, n: int, device) -> Tuple[torch.Tensor, torch.Tensor]:
    k1, k2 = _keys(seed, tid)
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    lo, hi = i & M32, i >> 32
    r1 = _hash32(_hash32(lo ^ k1) ^ _hash32(hi ^ k2))
    r2 = _hash32(r1 ^ k2)
    return r1, r2


CHUNK = 1 << 24


def normal_(out: torch.Tensor, seed: int, tid: int, std: float, start: int = 0) -> torch.Tensor:
    """Fill contiguous ``out`` (any float dtype, any device) with element
    ``start + j`` of stream ``(seed, tid)`` times ``std``."""
    flat = out.view(-1)
    n = flat.numel()
    for c0 in range(0, n, CHUNK):
        c1 = min(n, c0 + CHUNK)
        r1, r2 = _words(seed, tid, start + c0, c1 - c0, flat.device)
        u1 = (r1.to(torch.float64) + 0.5) * (1.0 / 4294967296.0)
        u2 = r2.to(torch.float64) * (1.0 / 4294967296.0)
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        flat[c0:c1] = (z * std).to(torch.float32).to(flat.dtype)
        del r1, r2, u1, u2, z
    return out


def normal(shape, seed: int, tid: int, std: float, dtype=torch.float32, device="cpu") -> torch.Tensor:
    t = torch.empty(shape, dtype=dtype, device=device)
    return normal_(t, seed, tid, std)


def permutation(n: int, seed: int, tid: int) -> List[int]:
    """A seeded permutation of 0..n-1 (sort of hashed keys; ties broken by index)."""
    k1, _ = _keys(seed, tid)
    keys = [(_hash32_int(_hash32_int(i ^ k1)), i) for i in range(n)]
    keys.sort()
    return [i for _, i in keys]


# ------------------------------------------------------------ configurations --

@dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int
    E: int
    k: int
    I: int
    gating: int
    shared: bool = False
    Ts: Tuple[int, ...] = ()
    skew: Optional[Tuple] = None      # None | ("normal", std) | ("zipf", s, beta)
    router_std: float = 0.02
    sel_bias_std: float = 0.0
    description: str = ""

    def with_T(self, T: int) -> "Workload":
        return Workload(self, T)


@dataclass(frozen=True)
class Workload:
    cfg: LayerConfig
    T: int

    @property
    def label(self) -> str:
        return f"{self.cfg.name}_T{self.T}"


CONFIGS: Dict[str, LayerConfig] = {
    "tiny": LayerConfig(
        "tiny", H=256, E=8, k=2, I=512, gating=GATE_TOPK_SOFTMAX, Ts=(64,),
        description="tiny MoE layer, 8 experts top-2, uniform routing"),
    "mixtral": LayerConfig(
        "mixtral", H=4096, E=8, k=2, I=14336, gating=GATE_TOPK_SOFTMAX,
        Ts=(1, 8, 64, 512, 4096), skew=("normal", 0.5),
        description="Mixtral-8x7B-shaped layer, per-expert logit offsets N(0,0.5^2)"),
    "qwen3": LayerConfig(
        "qwen3", H=4096, E=128, k=8, I=1536, gating=GATE_SOFTMAX_TOPK_RENORM,
        Ts=(1, 16, 128, 256, 1024), skew=("zipf", 1.1, ZIPF_BETA_QWEN3),
        description="Qwen3-235B-A22B-shaped layer, Zipf(1.1) logit skew"),
    "dsv3": LayerConfig(
        "dsv3", H=7168, E=256, k=8, I=2048, gating=GATE_SIGMOID_BIAS_RENORM, shared=True,
        Ts=(2048, 8192), skew=("zipf", 1.2, 1.0), sel_bias_std=0.1,
        description="DeepSeek-V3-shaped layer, 256 routed + 1 shared, Zipf(1.2) skew"),
    "qwen3_tp8": LayerConfig(
        "qwen3_tp8", H=4096, E=128, k=8, I=192, gating=GATE_SOFTMAX_TOPK_RENORM,
        Ts=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048), skew=("zipf", 1.1, ZIPF_BETA_QWEN3),
        description="one tensor-parallel rank (I/8=192) of the Qwen3-235B-A22B layer"),
}


def uniform_variant(cfg: LayerConfig) -> LayerConfig:
    """The same layer with no routing skew (delta = 0)."""
    return LayerConfig(cfg.name + "_uniform", cfg.H, cfg.E, cfg.k, cfg.I, cfg.gating, cfg.shared,
                       cfg.Ts, None, cfg.router_std, cfg.sel_bias_std, cfg.description + " (uniform)")


def logit_offsets(cfg: LayerConfig, seed: int) -> Optional[List[float]]:
    """Per-expert logit offsets delta_e of the configuration (None if uniform)."""
    if cfg.skew is None:
        return None
    if cfg.skew[0] == "normal":
        d = normal((cfg.E,), seed, TID_DELTA, float(cfg.skew[1]), torch.float64)
        return [float(v) for v in d]
    if cfg.skew[0] == "zipf":
        s, beta = float(cfg.skew[1]), float(cfg.skew[2])
        order = permutation(cfg.E, seed, TID_PERM)      # order[r] = expert of rank r+1
        delta = [0.0] * cfg.E
        for r, e in enumerate(order):
            delta[e] = -beta * s * math.log(r + 1)
        return delta
    raise ValueError(f"unknown skew {cfg.skew}")


@dataclass
class LayerInputs:
    cfg: LayerConfig
    T: int
    seed: int
    x: torch.Tensor                 # [T,H] bf16
    w_router: torch.Tensor          # [E,H] fp32
    sel_bias: Optional[torch.Tensor]   # [E] fp32 or None
    w13: torch.Tensor               # [E,2I,H] bf16
    w2: torch.Tensor                # [E,H,I] bf16
    w13_shared: Optional[torch.Tensor] = None   # [2I,H] bf16
    w2_shared: Optional[torch.Tensor] = None    # [H,I] bf16
    delta: Optional[List[float]] = field(default=None)


def make_tokens(cfg: LayerConfig, T: int, seed: int, device="cpu") -> torch.Tensor:
    x = normal((T, cfg.H), seed, TID_X, 1.0, torch.bfloat16, device)
    if cfg.skew is not None:
        x[:, 0] = 1.0
    return x


def make_router(cfg: LayerConfig, seed: int, device="cpu") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    w_r = normal((cfg.E, cfg.H), seed, TID_WR, cfg.router_std, torch.float32, device)
    delta = logit_offsets(cfg, seed)
    if delta is not None:
        w_r[:, 0] = torch.tensor(delta, dtype=torch.float64).to(torch.float32).to(device)
    b = None
    if cfg.gating == GATE_SIGMOID_BIAS_RENORM:
        b = normal((cfg.E,), seed, TID_BIAS, cfg.sel_bias_std, torch.float32, device)
    return w_r, b


def make_layer(cfg: LayerConfig, T: int, seed: int = 0, device="cpu") -> LayerInputs:
    H, E, I = cfg.H, cfg.E, cfg.I
    x = make_tokens(cfg, T, seed, device)
    w_r, b = make_router(cfg, seed, device)
    w13 = normal((E, 2 * I, H), seed, TID_W13, 1.0 / math.sqrt(H), torch.bfloat16, device)
    w2 = normal((E, H, I), seed, TID_W2, 1.0 / math.sqrt(I), torch.bfloat16, device)
    w13s = w2s = None
    if cfg.shared:
        w13s = normal((2 * I, H), seed, TID_W13S, 1.0 / math.sqrt(H), torch.bfloat16, device)
        w2s = normal((H, I), seed, TID_W2S, 1.0 / math.sqrt(I), torch.bfloat16, device)
    return LayerInputs(cfg, T, seed, x, w_r, b, w13, w2, w13s, w2s, logit_offsets(cfg, seed))


def random_ids(T: int, k: int, E: int, seed: int, tid: int = 11) -> torch.Tensor:
    """[T,k] int32 expert ids, k distinct per token, uniform (for dispatch tests)."""
    if k > E:
        raise ValueError("k > E")
    r = normal((T, E), seed, tid, 1.0, torch.float64)
    return torch.argsort(r, dim=1)[:, :k].to(torch.int32).contiguous()


def skewed_ids(T: int, k: int, E: int, seed: int, hot: int, tid: int = 12) -> torch.Tensor:
    """[T,k] ids where expert ``hot`` is in every token's set (maximal skew)."""
    ids = random_ids(T, k, E, seed, tid).clone()
    for t in range(T):
        row = ids[t].tolist()
        if hot not in row:
            row[-1] = hot
        ids[t] = torch.tensor(row, dtype=torch.int32)
    return ids
