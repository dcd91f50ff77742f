"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""

from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np
import torch

import oracle
import routed_expert_ffn_gb300 as moe
import synth

# Tolerances (stated with the layer configurations): routing metadata is
# bit-exact except at near-ties (top-k boundary gap below 1e-5); layer outputs
# reach relative L2 <= 1e-2 and per-element |err| <= 3e-2 * rms(y).
NEAR_TIE = 1e-5
REL_L2 = 1e-2
ELEM = 3e-2
GATE_ATOL = 1e-5


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_output_close(got: np.ndarray, ref: np.ndarray, what: str = "y"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = math.sqrt(float(np.mean(ref ** 2)))
    r = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert r <= REL_L2, f"{what}: relative L2 {r:.3e} > {REL_L2}"
    assert m <= ELEM * rms, f"{what}: max |err| {m:.3e} > {ELEM} * rms {rms:.3e}"
    return r, m / max(rms, 1e-300)


def assert_rows_close(got: np.ndarray, ref: np.ndarray, what: str = "rows"):
    """The output criterion applied to each row on its own scale: every row of
    out_perm is one expert's (gate-weighted) output, an output of its own."""
    worst = (0.0, 0.0)
    for i in range(ref.shape[0]):
        r, m = assert_output_close(got[i], ref[i], f"{what}[{i}]")
        worst = (max(worst[0], r), max(worst[1], m))
    return worst


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def selection_keys(s: np.ndarray, gating: int, bias: Optional[np.ndarray]) -> np.ndarray:
    """float32 selection keys per the gating variant (for validity checks)."""
    if gating == synth.GATE_SIGMOID_BIAS_RENORM:
        a = (1.0 / (1.0 + np.exp(-s.astype(np.float64)))).astype(np.float32)
        return (a + bias.astype(np.float32)).astype(np.float32)
    return s.astype(np.float32)


# Routing counts of every check_routing call in this session, printed in the
# terminal summary (tests/conftest.py): the configuration statement asks for
# near-ties to be counted and reported, not only tolerated.
ROUTING_REPORT = []


def check_routing(gpu_ids: np.ndarray, gpu_w: np.ndarray, ref: Dict[str, np.ndarray], gating: int,
                  bias, label: str = "") -> Dict[str, int]:
    """Routing parity.  Off near-ties (oracle boundary gap >= NEAR_TIE) the
    selected expert set is bit-exact and each expert's gate weight is within
    GATE_ATOL.  Slot order is exact too, except that two selected experts whose
    oracle keys differ by less than NEAR_TIE may take each other's slot: fp32
    logits carry about 1.2e-5 of rounding at these magnitudes, so the order of
    near-equal keys is not unique; every such slot difference is counted
    (order_swaps).  On near-tie tokens the GPU's set must be a valid top-k of
    the oracle's keys within NEAR_TIE; a different but valid set is counted
    (flips).  The counts are returned and recorded in ROUTING_REPORT."""
    T, k = gpu_ids.shape
    gap = ref["gap"]
    keys = selection_keys(ref["logits"], gating, None if bias is None else np.asarray(bias))
    clear = ~(gap < NEAR_TIE)          # NaN gap (k == E) counts as clear
    g_sorted = np.sort(gpu_ids, axis=1)
    r_sorted = np.sort(ref["ids"], axis=1)
    assert np.array_equal(g_sorted[clear], r_sorted[clear]), "selected experts differ off near-ties"
    # gate weight of each selected expert (matched by expert id)
    go, ro = np.argsort(gpu_ids, axis=1), np.argsort(ref["ids"], axis=1)
    gw = np.take_along_axis(gpu_w, go, 1)
    rw = np.take_along_axis(ref["w"], ro, 1)
    assert np.max(np.abs(gw[clear] - rw[clear]), initial=0.0) <= GATE_ATOL
    # slot order: non-increasing oracle keys up to near-equal keys
    kg = np.take_along_axis(keys, gpu_ids.astype(np.int64), 1).astype(np.float64)
    assert np.all(np.diff(kg, axis=1) <= NEAR_TIE), "slots not in best-first order"
    # off near-ties, a slot may differ from the oracle's only between experts
    # whose keys are within NEAR_TIE of each other
    kr = np.take_along_axis(keys, ref["ids"].astype(np.int64), 1).astype(np.float64)
    slot_diff = clear[:, None] & (gpu_ids != ref["ids"])
    assert np.all(np.abs(kg - kr)[slot_diff] < NEAR_TIE), "slot order differs at a clear key gap"
    swaps = int(np.sum(np.any(slot_diff, axis=1)))
    ties = np.where(~clear)[0]
    flips = 0
    for t in ties:
        kth = np.sort(keys[t])[::-1][k - 1]
        sel = set(gpu_ids[t].tolist())
        assert len(sel) == k
        for e in range(keys.shape[1]):
            if e in sel:
                assert keys[t, e] >= kth - NEAR_TIE
            else:
                assert keys[t, e] <= kth + NEAR_TIE
        flips += int(set(gpu_ids[t].tolist()) != set(ref["ids"][t].tolist()))
    info = {"tokens": int(T), "near_ties": int(len(ties)), "flips": flips, "order_swaps": swaps}
    ROUTING_REPORT.append((label or f"T={T}", info))
    return info


class LayerRun:
    """One moe_layer_forward of a seeded workload on cuda:0."""

    def __init__(self, inputs: synth.LayerInputs, path: Optional[int] = None):
        cfg, T = inputs.cfg, inputs.T
        self.inputs = inputs
        self.path = path     # None: moe_layer_forward's own choice; else MOE_PATH_*
        self.d = moe.desc(T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gating, cfg.shared)
        self.ws = moe.alloc_workspace(self.d)
        self.layout = moe.moe_workspace_layout(self.d)
        self.w = moe.layer_weights(inputs.w_router, inputs.w13, inputs.w2, inputs.sel_bias,
                                   inputs.w13_shared, inputs.w2_shared)
        self.y = torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")

    def forward(self):
        moe.moe_layer_forward(self.d, self.w, self.inputs.x, self.y, self.ws, path=self.path)
        torch.cuda.synchronize()
        st, raw = moe.moe_get_device_status(self.ws)
        assert st == moe.MOE_OK, (st, raw)
        return self.y

    def view(self, name, dtype, shape):
        return moe.workspace_view(self.ws, self.layout, name, dtype, shape)

    def metadata(self):
        cfg, T = self.inputs.cfg, self.inputs.T
        Na = T * cfg.k
        g = lambda n, dt, sh: self.view(n, dt, sh).cpu().numpy()
        return {
            "logits": g("logits", torch.float32, (T, cfg.E)),
            "ids": g("topk_ids", torch.int32, (T, cfg.k)),
            "w": g("topk_w", torch.float32, (T, cfg.k)),
            "gap": g("gap", torch.float32, (T,)),
            "counts": g("counts", torch.int32, (cfg.E,)),
            "offsets": g("offsets", torch.int32, (cfg.E + 1,)),
            "perm_src": g("perm_src", torch.int32, (Na,)),
            "inv_pos": g("inv_pos", torch.int32, (Na,)),
            "w_perm": g("w_perm", torch.float32, (Na,)),
        }


def host_copy(inputs: synth.LayerInputs, experts: Optional[Sequence[int]] = None):
    """Host copies of the exact bytes the GPU used: x, router, bias, and the
    listed experts' weight blocks (all experts when None)."""
    E = inputs.cfg.E
    ex = range(E) if experts is None else experts
    return {
        "x": inputs.x.cpu(),
        "w_router": inputs.w_router.cpu(),
        "sel_bias": None if inputs.sel_bias is None else inputs.sel_bias.cpu(),
        "w13": {e: inputs.w13[e].cpu() for e in ex},
        "w2": {e: inputs.w2[e].cpu() for e in ex},
        "w13_shared": None if inputs.w13_shared is None else inputs.w13_shared.cpu(),
        "w2_shared": None if inputs.w2_shared is None else inputs.w2_shared.cpu(),
    }


def segment_edge_tokens(perm_src: np.ndarray, offsets: np.ndarray, e: int, k: int,
                        step: int = 128) -> set:
    """Tokens at the first and last row of every `step`-row chunk of expert
    e's segment (positions 0, step-1, step, 2*step-1, ... and the last row):
    the boundaries of the GEMMs' 128-row token chunks and of both 128-row
    halves of their 256-row tiles."""
    lo, hi = int(offsets[e]), int(offsets[e + 1])
    m = hi - lo
    pos = set()
    for c in range(0, m, step):
        pos.add(c)
        pos.add(min(c + step - 1, m - 1))
    return {int(perm_src[lo + p]) // k for p in pos}


def sample_tokens(T: int, n: int, ids: np.ndarray, counts: np.ndarray, seed: int = 0,
                  perm_src: Optional[np.ndarray] = None, offsets: Optional[np.ndarray] = None,
                  shared: bool = False):
    """A seeded token sample of at least min(n, T) tokens.  It always holds the
    first and last token, a token of the hottest and of the coldest touched
    expert, and -- given the dispatch layout -- the tokens at the first and
    last row of every 128-row chunk of the two hottest experts' segments and
    of the shared expert's segment (all T tokens in order)."""
    if T <= n:
        return list(range(T))
    k = ids.shape[1]
    pick = {0, T - 1}
    touched = np.where(counts > 0)[0]
    order = touched[np.argsort(-counts[touched], kind="stable")]
    hot, cold = int(order[0]), int(order[-1])
    for e in (hot, cold):
        rows = np.where((ids == e).any(axis=1))[0]
        pick.add(int(rows[0]))
        pick.add(int(rows[-1]))
    if perm_src is not None and offsets is not None:
        for e in order[:2]:
            pick |= segment_edge_tokens(perm_src, offsets, int(e), k)
    if shared:
        for c in range(0, T, 128):
            pick.add(c)
            pick.add(min(c + 127, T - 1))
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(pick, dtype=np.int64))
    need = max(0, n - len(pick))
    if need:
        pick |= set(rng.choice(rest, size=min(need, rest.size), replace=False).tolist())
    return sorted(int(t) for t in pick)
