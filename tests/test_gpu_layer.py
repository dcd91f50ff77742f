"""Whole-layer parity of moe_layer_forward with the CPU oracle on the five
layer configurations (needs a GB300).

Small batches are checked on every token; large ones on a seeded sample of at
least 256 tokens that holds the first and last row of every 128-row chunk of
the two hottest experts and of the shared expert (the GEMMs' token-chunk
boundaries and both halves of their 256-row tiles), a token of the coldest
touched expert, and seeded random tokens.
Routing metadata is compared on all tokens: ids bit-exact off near-ties, and
counts / offsets / permutation / inverse bit-exact against the oracle's
dispatch of the same ids."""

import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_gb300 as moe
import synth
from gpu_check import LayerRun, assert_output_close, bf16_np, check_routing, host_copy, sample_tokens

pytestmark = pytest.mark.gpu

_WEIGHTS = {}


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    _WEIGHTS.clear()
    torch.cuda.empty_cache()


def layer_inputs(name, T, seed=0, uniform=False):
    """Seeded inputs on cuda:0; the expert weights are generated once per
    configuration and shared by its batch sizes."""
    cfg = synth.CONFIGS[name]
    if uniform:
        cfg = synth.uniform_variant(cfg)
    key = (name, seed)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        torch.cuda.empty_cache()
        full = synth.make_layer(cfg, 1, seed, device="cuda")
        _WEIGHTS[key] = full
    full = _WEIGHTS[key]
    x = synth.make_tokens(cfg, T, seed, device="cuda")
    w_r, b = synth.make_router(cfg, seed, device="cuda")
    return synth.LayerInputs(cfg, T, seed, x, w_r, b, full.w13, full.w2, full.w13_shared,
                             full.w2_shared)


def check_layer(inputs, n_sample=256, path=None):
    cfg, T = inputs.cfg, inputs.T
    run = LayerRun(inputs, path)
    y = run.forward()
    meta = run.metadata()
    host = host_copy(inputs, experts=[])
    s = oracle.router_logits(host["x"], host["w_router"])
    ids, w, gap = oracle.topk_gating(s, cfg.k, cfg.gating, host["sel_bias"])
    ref = {"logits": s, "ids": ids, "w": w, "gap": gap}
    bias = None if host["sel_bias"] is None else host["sel_bias"].numpy()
    info = check_routing(meta["ids"], meta["w"], ref, cfg.gating, bias,
                         label=f"{cfg.name} T={T}" + ("" if path is None else f" path={path}"))
    # dispatch of the ids the GPU routed (a pure integer function of them)
    rc, ro, rp, ri = oracle.dispatch(meta["ids"], cfg.E)
    assert np.array_equal(meta["counts"], rc)
    assert np.array_equal(meta["offsets"], ro)
    assert np.array_equal(meta["perm_src"], rp)
    assert np.array_equal(meta["inv_pos"], ri)
    assert np.array_equal(meta["w_perm"], meta["w"].reshape(-1)[rp])
    # outputs on the sampled tokens whose routing is not a near-tie
    toks = sample_tokens(T, n_sample, meta["ids"], rc, perm_src=meta["perm_src"],
                         offsets=meta["offsets"], shared=bool(cfg.shared))
    toks = [t for t in toks if not (ref["gap"][t] < 1e-5)]
    need = sorted({int(e) for t in toks for e in ref["ids"][t]})
    host = host_copy(inputs, experts=need)
    y_ref = oracle.layer_tokens(host["x"], ref["ids"], ref["w"], host["w13"], host["w2"], toks,
                                host["w13_shared"], host["w2_shared"])
    got = bf16_np(y[toks])
    r, m = assert_output_close(got, y_ref)
    num, den = oracle.imbalance(rc, T * cfg.k)
    return {"rel_l2": r, "max_rel": m, "imbalance": num / den, "checked_tokens": len(toks),
            **info}


@pytest.mark.parametrize("T", [64, 1, 17])
def test_tiny_layer(T):
    check_layer(layer_inputs("tiny", T), n_sample=64)


@pytest.mark.parametrize("T", [1, 8, 64, 512, 4096])
def test_mixtral_layer(T):
    info = check_layer(layer_inputs("mixtral", T))
    assert info["checked_tokens"] >= min(T, 256)


@pytest.mark.parametrize("T", [1, 16, 128, 256, 1024])
def test_qwen3_layer(T):
    info = check_layer(layer_inputs("qwen3", T), n_sample=128)
    if T == 1024:
        assert 2.7 <= info["imbalance"] <= 3.3


def test_qwen3_layer_uniform_routing():
    check_layer(layer_inputs("qwen3", 1024, uniform=True), n_sample=64)


@pytest.mark.parametrize("T", [1, 8, 64, 256, 2048])
def test_qwen3_tp8_slice_layer(T):
    check_layer(layer_inputs("qwen3_tp8", T), n_sample=128)


@pytest.mark.parametrize("T", [2048, 8192])
def test_dsv3_layer(T):
    info = check_layer(layer_inputs("dsv3", T))
    assert info["checked_tokens"] >= 256


def test_output_independent_of_batch_neighbours():
    # dropless: a token's output does not depend on the rest of the batch
    big = layer_inputs("qwen3", 256)
    y_big = LayerRun(big).forward().clone()
    for t in (0, 99, 255):
        one = synth.LayerInputs(big.cfg, 1, 0, big.x[t:t + 1].contiguous(), big.w_router, None,
                                big.w13, big.w2)
        y1 = LayerRun(one).forward()
        assert_output_close(bf16_np(y1[0]), bf16_np(y_big[t]), "batch independence")


def _split_kbs(total, nkb, num_sms, max_m):
    """K blocks per split-K piece, by the rule the tile plan documents: split only
    when every tile has <= 32 token rows and the busiest SM's K blocks (plus a
    fixed cost of 8 K blocks per piece, plus the pieces) drop by at least a fifth;
    pieces are even numbers of K blocks."""
    if total <= 0 or max_m > 32 or total > 512:
        return nkb
    base = -(-total // num_sms) * nkb
    best, best_cost = nkb, base
    for S in range(2, 17):
        kbs = 2 * (-(-nkb // (2 * S)))
        if kbs >= nkb:
            continue
        pieces = -(-nkb // kbs)
        if total * pieces > 1024:
            break
        cost = -(-(total * pieces) // num_sms) * (kbs + 8) + pieces
        if cost < best_cost:
            best, best_cost = kbs, cost
    return best if best_cost * 5 <= base * 4 else nkb


@pytest.mark.parametrize("name,T", [("qwen3", 1), ("qwen3", 256), ("qwen3", 1024),
                                    ("mixtral", 4096), ("qwen3_tp8", 8), ("dsv3", 8192)])
def test_tile_plan(name, T):
    """The device-side tile plan (segments, tile prefixes, split-K pieces, layouts)
    is an integer function of the dispatch counts: recomputed here from the rules
    and compared exactly."""
    inputs = layer_inputs(name, T)
    cfg = inputs.cfg
    run = LayerRun(inputs, moe.MOE_PATH_KERNEL_CHAIN)   # the plan drives the chain's GEMMs
    run.forward()
    counts = run.metadata()["counts"].tolist()
    ms = counts + ([T] if cfg.shared else [])
    nseg = len(ms)
    plan = run.view("plan", torch.int32, (3 * (nseg + 1) + 4,)).cpu().numpy().tolist()
    cdiv = lambda a, b: -(-a // b)
    Na = T * cfg.k
    seg_row = np.concatenate([[0], np.cumsum(counts)]).tolist()[:cfg.E]
    if cfg.shared:
        seg_row.append(Na)
    seg_row.append(Na + (T if cfg.shared else 0))
    live = [m for m in ms if m > 0]
    n_chunks = sum(cdiv(m, 256) for m in live)
    n_wide = sum(m // 256 + (1 if m % 256 > 128 else 0) for m in live)
    st_narrow = sum(cdiv(m, 128) for m in live)
    st_wide = sum(2 * cdiv(m, 256) for m in live)
    wide_dn = n_wide > 0 and 2 * n_wide >= n_chunks
    wide_gu = st_narrow > 0 and 8 * st_wide <= 9 * st_narrow
    # gate/up tiles per segment: wide (64+64 rows by <= 256 tokens) above
    # wide_above rows, else 128+128 rows by <= 128 tokens
    wide_above = 0 if wide_gu else (1 << 30 if max(ms) <= 16 else 1024)
    gu = [cdiv(m, 256) * cdiv(cfg.I, 64) if m > wide_above else cdiv(m, 128) * cdiv(cfg.I, 128)
          for m in ms]
    # down: "pair" tiles (256 W2 rows by <= 128 token rows) where the launch
    # would otherwise be narrow or medium
    pair = max(ms) > 16 and not wide_dn and cfg.H >= 256
    # the same tiles in the thin layout when the down K is short
    thin_pair = max(ms) <= 16 and cfg.H >= 256 and cfg.I <= 4096
    dn = [cdiv(m, 128) * cdiv(cfg.H, 256) if pair or thin_pair
          else cdiv(m, 256) * cdiv(cfg.H, 128) for m in ms]
    pref = lambda v: np.concatenate([[0], np.cumsum(v)]).astype(int).tolist()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    want = (seg_row + pref(gu) + pref(dn) +
            [_split_kbs(sum(gu), cfg.H // 64, nsm, max(ms)),
             _split_kbs(sum(dn), cfg.I // 64, nsm, max(ms))])
    # pipeline layouts: 2 = thin (every segment <= 16 rows), 3 = medium (down, <= 64),
    # 1 = wide, 4 = pair (down), 5 = thin pair (down), 0 = narrow
    thin = max(ms) <= 16
    medium = max(ms) <= 64
    want += [2 if thin else int(wide_gu),
             (5 if thin_pair else 2) if thin else
             (4 if pair else (3 if medium else (1 if wide_dn else 0)))]
    assert plan == want
    if name == "mixtral":
        assert wide_gu and wide_dn   # uniform prefill: both GEMMs run wide
    if (name, T) == ("qwen3", 1024):
        assert not wide_gu and not wide_dn and pair
    if (name, T) in (("qwen3", 1), ("qwen3_tp8", 8)):
        assert thin
    if (name, T) == ("qwen3", 256):
        assert medium and not thin and pair   # the pair layout takes the medium batches
