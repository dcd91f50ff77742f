"""moe_build_dispatch_noalloc, the dispatch entry point for callers that
cannot allocate device memory (a plugin inside a framework that owns the
device-memory budget, a path that must not risk cudaMalloc's device
synchronisation): its scratch is a fixed array inside the library instead of a
caller workspace.  Its results must equal moe_build_dispatch's bit for bit, on
consecutive calls that reuse the shared array.  This file is collected last so
that a run stopping at the first failure has run every other test first."""

import numpy as np
import pytest
import torch

import routed_expert_ffn_gb300 as moe
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from routed_expert_ffn_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _outputs(T, k, E):
    z = lambda n, dt: torch.empty(n, dtype=dt, device="cuda")
    return (z(E, torch.int32), z(E + 1, torch.int32), z(T * k, torch.int32), z(T * k, torch.int32),
            z(T * k, torch.float32))


def _with_workspace(ids, w, E):
    T, k = ids.shape
    d = moe.desc(T, 64, E, k, 64, 0)
    ws = moe.alloc_workspace(d)
    out = _outputs(T, k, E)
    moe.moe_build_dispatch(d, ids, w, *out, ws)
    st, _ = moe.moe_get_device_status(ws)
    return st, [o.cpu() for o in out]


def _without_workspace(ids, w, E):
    T, k = ids.shape
    d = moe.desc(T, 64, E, k, 64, 0)
    out = _outputs(T, k, E)
    if w is None:
        out = out[:4] + (None,)          # no gate weights to permute
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_build_dispatch_noalloc(d, ids, w, *out, status)
    torch.cuda.synchronize()
    return int(status.item()), [o.cpu() for o in out if o is not None]


# two calls in a row with different shapes: the second reuses the array the
# first one left behind
CASES = [[(8192, 8, 256, True), (1024, 8, 128, False)],
         [(4096, 2, 8, False), (333, 4, 64, True)]]


@pytest.mark.parametrize("calls", CASES)
def test_noalloc_dispatch_matches_workspace_dispatch(calls):
    for T, k, E, skew in calls:
        ids = (synth.skewed_ids(T, k, E, T, hot=E // 2) if skew else
               synth.random_ids(T, k, E, T)).cuda()
        w = synth.normal((T, k), T, 7, 1.0, torch.float32).cuda()
        st_ws, ref = _with_workspace(ids, w, E)
        st_na, got = _without_workspace(ids, w, E)
        assert st_ws == moe.MOE_OK and st_na == 0
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_reports_bad_ids_and_rejects_oversize():
    ids = synth.random_ids(100, 2, 8, 0)
    ids[3, 1] = 9
    st, _ = _without_workspace(ids.cuda(), None, 8)
    assert st & 1
    # a batch whose tables exceed the fixed array is refused before any launch
    T, k, E = 65536 // 8 + 32, 8, 512
    d = moe.desc(T, 64, E, k, 64, 0)
    out = _outputs(T, k, E)
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_build_dispatch_noalloc(d, ids, None, *out[:4], None)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE


def test_noalloc_reserves_no_device_memory_after_the_first_call():
    # The first call on a device may make the CUDA runtime load this library's
    # device code and reserve the fixed array (lazy module loading); after it,
    # calls of any accepted shape reserve nothing: the device's free memory
    # does not move.  All outputs are allocated before the first reading.
    shapes = [(4096, 8, 256), (17, 2, 8), (1024, 8, 128), (3000, 32, 64)]
    bufs = []
    for T, k, E in shapes:
        ids = synth.random_ids(T, k, E, T).cuda()
        w = synth.normal((T, k), T, 7, 1.0, torch.float32).cuda()
        bufs.append((moe.desc(T, 64, E, k, 64, 0), ids, w, _outputs(T, k, E)))
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    d, ids, w, out = bufs[0]
    moe.moe_build_dispatch_noalloc(d, ids, w, *out, status)   # warm-up call
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for rep in range(3):
        for d, ids, w, out in bufs:
            moe.moe_build_dispatch_noalloc(d, ids, w, *out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.cuda.mem_get_info()[0] == free0, rep
