"""Parity of each C ABI stage call with the CPU oracle (needs a GB300)."""

import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_gb300 as moe
import synth
from conftest import golden
from gpu_check import (GATE_ATOL, NEAR_TIE, assert_output_close, assert_rows_close, bf16_np,
                       check_routing)

pytestmark = pytest.mark.gpu

MODES = [synth.GATE_TOPK_SOFTMAX, synth.GATE_SOFTMAX_TOPK, synth.GATE_SOFTMAX_TOPK_RENORM,
         synth.GATE_SIGMOID_BIAS_RENORM]


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _route_gpu(d, x, w_r, b):
    T, E, k = d.T, d.E, d.k
    ws = moe.alloc_workspace(d)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    gap = torch.empty((T,), dtype=torch.float32, device="cuda")
    moe.moe_route(d, x, w_r, b, logits, ids, w, gap, ws)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy()


# ------------------------------------------------------------------ route --

def test_route_page_example_all_modes():
    kv, _ = golden("router_8expert_top2.txt")
    scores = [float(v) for v in kv["scores"]]
    H, E = 256, 8
    x = torch.zeros((1, H), dtype=torch.bfloat16)
    x[0, 0] = 1.0
    w_r = synth.normal((E, H), 3, 99, 0.5, torch.float32)
    w_r[:, 0] = torch.tensor(scores)
    for mode in MODES:
        d = moe.desc(1, H, E, 2, 64, mode)
        b = torch.zeros(E, dtype=torch.float32, device="cuda")
        s, ids, w, gap = _route_gpu(d, x.cuda(), w_r.cuda(), b)
        assert np.array_equal(s[0], np.array(scores, dtype=np.float32))
        assert ids[0].tolist() == [1, 4]
        ref_ids, ref_w, _ = oracle.topk_gating(s, 2, mode, np.zeros(E, np.float32))
        assert np.max(np.abs(w - ref_w)) <= GATE_ATOL


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,H,E,k", [(1, 256, 8, 2), (37, 256, 8, 1), (200, 512, 64, 6),
                                     (130, 1024, 128, 8), (64, 256, 256, 8), (33, 256, 512, 32),
                                     (5, 256, 4, 4), (300, 4096, 128, 8)])
def test_route_matches_oracle(mode, T, H, E, k):
    seed = T + E + k + mode
    x = synth.normal((T, H), seed, 1, 1.0, torch.bfloat16)
    w_r = synth.normal((E, H), seed, 2, 0.05, torch.float32)
    b = synth.normal((E,), seed, 3, 0.1, torch.float32)
    d = moe.desc(T, H, E, k, 64, mode)
    s, ids, w, gap = _route_gpu(d, x.cuda(), w_r.cuda(), b.cuda())
    rs = oracle.router_logits(x, w_r)
    r_ids, r_w, r_gap = oracle.topk_gating(rs, k, mode, b)
    assert np.max(np.abs(s - rs)) <= 1e-4 * max(1.0, float(np.max(np.abs(rs))))
    info = check_routing(ids, w, {"ids": r_ids, "w": r_w, "gap": r_gap, "logits": rs}, mode, b.numpy(),
                         label=f"route mode={mode} T={T} E={E} k={k}")
    if k < E:
        clear = ~(r_gap < NEAR_TIE)
        assert np.allclose(gap[clear], r_gap[clear], atol=1e-5, rtol=0)
    else:
        assert np.all(gap == 0)
    assert info["flips"] <= max(1, T // 100)


# --------------------------------------------------------------- dispatch --

def _dispatch_gpu(ids_np, E, w_np=None):
    T, k = ids_np.shape
    d = moe.desc(T, 64, E, k, 64, 0)
    ws = moe.alloc_workspace(d)
    ids = torch.from_numpy(np.ascontiguousarray(ids_np)).cuda()
    w = None if w_np is None else torch.from_numpy(np.ascontiguousarray(w_np)).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    wp = None if w is None else torch.empty(T * k, dtype=torch.float32, device="cuda")
    moe.moe_build_dispatch(d, ids, w, counts, offsets, perm, inv, wp, ws)
    st, raw = moe.moe_get_device_status(ws)
    out = [a.cpu().numpy() for a in (counts, offsets, perm, inv)]
    return st, out, (None if wp is None else wp.cpu().numpy())


def test_dispatch_page_example():
    kv, _ = golden("dispatch_5token.txt")
    ids = np.array([int(v) for v in kv["ids"]], dtype=np.int32).reshape(-1, 1)
    st, (counts, offsets, perm, inv), _ = _dispatch_gpu(ids, int(kv["E"][0]))
    assert st == moe.MOE_OK
    assert counts.tolist() == [int(v) for v in kv["counts"]]
    assert perm.tolist() == [3, 1, 0, 2, 4]
    assert inv.tolist() == [2, 1, 3, 0, 4]


@pytest.mark.parametrize("T,k,E,skew", [(1, 1, 1, False), (1, 8, 128, False), (37, 2, 8, False),
                                        (1024, 8, 128, False), (1024, 8, 128, True),
                                        (513, 8, 512, False), (8192, 8, 256, True),
                                        (4096, 2, 8, False), (3000, 32, 64, False)])
def test_dispatch_bit_exact(T, k, E, skew):
    ids = (synth.skewed_ids(T, k, E, T, hot=E // 3) if skew else synth.random_ids(T, k, E, T)).numpy()
    w = synth.normal((T, k), T, 7, 1.0, torch.float32).numpy()
    st, (counts, offsets, perm, inv), wp = _dispatch_gpu(ids, E, w)
    assert st == moe.MOE_OK
    rc, ro, rp, ri = oracle.dispatch(ids, E)
    assert np.array_equal(counts, rc)
    assert np.array_equal(offsets, ro)
    assert np.array_equal(perm, rp)
    assert np.array_equal(inv, ri)
    assert np.array_equal(wp, w.reshape(-1)[rp])


def test_dispatch_flags_bad_ids():
    ids = synth.random_ids(100, 2, 8, 0).numpy()
    ids[17, 1] = 8
    ids[50, 0] = -3
    st, _, _ = _dispatch_gpu(ids, 8)
    assert st == moe.MOE_ERR_DEVICE_CHECK


# ---------------------------------------------------- grouped FFN, combine --

def _ffn_case(T, H, I, E, k, seed, shared=False, skew=False):
    x = synth.normal((T, H), seed, 1, 1.0, torch.bfloat16)
    w13 = synth.normal((E, 2 * I, H), seed, 4, H ** -0.5, torch.bfloat16)
    w2 = synth.normal((E, H, I), seed, 5, I ** -0.5, torch.bfloat16)
    w13s = w2s = None
    if shared:
        w13s = synth.normal((2 * I, H), seed, 6, H ** -0.5, torch.bfloat16)
        w2s = synth.normal((H, I), seed, 7, I ** -0.5, torch.bfloat16)
    ids = (synth.skewed_ids(T, k, E, seed, hot=1) if skew else synth.random_ids(T, k, E, seed))
    # positive gate weights that sum to 1 per token, as every renormalising
    # gating variant produces
    w = torch.abs(synth.normal((T, k), seed, 8, 1.0, torch.float32)) + 0.05
    w = (w / w.sum(dim=1, keepdim=True)).contiguous()
    return x, w13, w2, w13s, w2s, ids, w


@pytest.mark.parametrize("T,H,I,E,k,shared,skew", [
    (1, 256, 512, 8, 2, False, False),        # decode: one row per expert
    (37, 256, 512, 8, 2, False, False),       # ragged rows, several weight blocks
    (300, 256, 256, 4, 2, False, True),       # an expert with > 128 rows: several token chunks
    (64, 384, 192, 16, 4, False, False),      # I = 192: ragged weight-row block, H not /128
    (20, 256, 256, 8, 2, True, False),        # shared expert segment
    (5, 128, 64, 2, 2, False, False),         # smallest shapes
])
def test_grouped_ffn_and_combine(T, H, I, E, k, shared, skew):
    x, w13, w2, w13s, w2s, ids, w = _ffn_case(T, H, I, E, k, seed=T + H + I, shared=shared, skew=skew)
    d = moe.desc(T, H, E, k, I, 0, shared)
    ws = moe.alloc_workspace(d)
    dev = lambda t: None if t is None else t.cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    wp = torch.empty(T * k, dtype=torch.float32, device="cuda")
    R = T * k + (T if shared else 0)
    out = torch.empty((R, H), dtype=torch.float16, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_build_dispatch(d, dev(ids), dev(w), counts, offsets, perm, inv, wp, ws)
    moe.moe_grouped_swiglu_ffn(d, dev(x), perm, offsets, wp, dev(w13), dev(w2), dev(w13s), dev(w2s),
                               out, ws)
    moe.moe_combine(d, out, inv, None, y)
    st, raw = moe.moe_get_device_status(ws)
    assert st == moe.MOE_OK, raw
    # out_perm row p = w[a] * FFN_e(x_t) for the assignment a at position p
    _, _, rp, _ = oracle.dispatch(ids.numpy(), E)
    ref = np.empty((R, H))
    idn, wn = ids.numpy(), w.numpy()
    for p, a in enumerate(rp):
        t, j = divmod(int(a), k)
        ref[p] = wn[t, j] * oracle.expert_ffn(x[t], w13[idn[t, j]], w2[idn[t, j]])
    for t in range(T if shared else 0):
        ref[T * k + t] = oracle.expert_ffn(x[t], w13s, w2s)
    assert_rows_close(out.double().cpu().numpy(), ref, "out_perm")
    # the layer output: combine of those rows
    y_ref = oracle.layer_tokens(x, idn, wn.astype(np.float64), w13, w2, range(T), w13s, w2s)
    assert_output_close(bf16_np(y), y_ref, "y")


def test_combine_exact_sum():
    # combine alone on given rows: the bf16 rounding of an fp32 sum
    T, k, H, E = 50, 4, 256, 16
    ids = synth.random_ids(T, k, E, 1).numpy()
    _, _, rp, ri = oracle.dispatch(ids, E)
    rows = synth.normal((T * k + T, H), 1, 9, 1.0, torch.float16)
    tw = synth.normal((T, k), 1, 10, 1.0, torch.float32)
    for shared in (False, True):
        d = moe.desc(T, H, E, k, 64, 0, shared)
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine(d, rows.cuda(), torch.from_numpy(ri).cuda(), tw.cuda(), y)
        torch.cuda.synchronize()
        r = rows.double().numpy()
        ref = np.zeros((T, H))
        for t in range(T):
            for j in range(k):
                ref[t] += tw[t, j].item() * r[ri[t * k + j]]
            if shared:
                ref[t] += r[T * k + t]
        got = bf16_np(y)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


def test_out_of_fp16_range_output_is_clamped_and_flagged():
    # an expert whose output exceeds the fp16 range of out_perm: the element is
    # clamped (never inf) and the status word reports a device check
    T, H, I, E, k = 8, 128, 64, 2, 1
    x, w13, w2, _, _, _, _ = _ffn_case(T, H, I, E, k, seed=3)
    w2 = (w2.float() * 1.0e6).to(torch.bfloat16)
    ids = torch.zeros((T, k), dtype=torch.int32)
    w = torch.ones((T, k), dtype=torch.float32)
    d = moe.desc(T, H, E, k, I, 0)
    ws = moe.alloc_workspace(d)
    z = lambda n, dt: torch.empty(n, dtype=dt, device="cuda")
    counts, offsets, perm, inv, wp = (z(E, torch.int32), z(E + 1, torch.int32), z(T * k, torch.int32),
                                      z(T * k, torch.int32), z(T * k, torch.float32))
    out = z((T * k, H), torch.float16)
    moe.moe_build_dispatch(d, ids.cuda(), w.cuda(), counts, offsets, perm, inv, wp, ws)
    moe.moe_grouped_swiglu_ffn(d, x.cuda(), perm, offsets, wp, w13.cuda(), w2.cuda(), None, None,
                               out, ws)
    st, raw = moe.moe_get_device_status(ws)
    assert st == moe.MOE_ERR_DEVICE_CHECK and raw & (1 << 5)
    o = out.float()
    assert torch.isfinite(o).all() and o.abs().max().item() == 65504.0
