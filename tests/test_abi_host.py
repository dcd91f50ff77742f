"""The C ABI on the host (no GPU): the library loads, exports every function
include/moe.h declares, sizes workspaces, and rejects bad arguments before it
launches anything."""

import ctypes
import os
import re

import pytest

import routed_expert_ffn_gb300 as moe
from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from routed_expert_ffn_gb300 import build
        build.build()
    return moe.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in ["moe_route", "moe_build_dispatch", "moe_grouped_swiglu_ffn", "moe_combine",
              "moe_layer_forward"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def qwen3(T=1024, **kw):
    d = dict(T=T, H=4096, E=128, k=8, I=1536, gating=moe.MOE_GATE_SOFTMAX_TOPK_RENORM, shared=False)
    d.update(kw)
    return moe.desc(**d)


def test_workspace_size_and_layout(lib):
    d = qwen3()
    n = moe.moe_workspace_size(d)
    lay = moe.moe_workspace_layout(d)
    assert n == lay["total"] > 0
    offs = sorted(v for k, v in lay.items() if k != "total")
    assert all(o % 1024 == 0 for o in offs)
    assert len(set(offs)) == len(offs)
    R = 1024 * 8
    assert lay["out_perm"] + R * 4096 * 2 <= n
    # the shared expert adds T rows to every permuted buffer
    ds = moe.desc(T=64, H=7168, E=256, k=8, I=2048, gating=3, shared=True)
    ls = moe.moe_workspace_layout(ds)
    assert ls["h"] - ls["x_perm"] >= (64 * 8 + 64) * 7168 * 2


@pytest.mark.parametrize("kw", [dict(T=0), dict(E=513), dict(k=0), dict(k=129), dict(k=33, E=64),
                                dict(H=4000), dict(I=1000), dict(H=32), dict(T=1 << 21)])
def test_bad_shapes(lib, kw):
    d = qwen3(**kw)
    assert moe.moe_workspace_size(d) == 0
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_layout(d)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE


def test_bad_enums(lib):
    for d in (qwen3(gating=4), qwen3(gating=-1), moe.LayerDesc(8, 256, 8, 2, 512, 0, 2)):
        assert moe.moe_workspace_size(d) == 0


FAKE = 1 << 20  # a 256-aligned non-null address; never dereferenced on the host


def test_route_validation_before_launch(lib):
    d = qwen3(T=16)
    n = moe.moe_workspace_size(d)
    P, S = ctypes.c_void_p, ctypes.c_size_t
    call = lambda **kw: lib.moe_route(ctypes.byref(kw.get("d", d)), kw.get("x", FAKE), FAKE, None,
                                      FAKE, FAKE, FAKE, None, kw.get("ws", FAKE),
                                      kw.get("n", n), None)
    assert call(x=None) == moe.MOE_ERR_INVALID_ARG
    assert call(x=FAKE + 4) == moe.MOE_ERR_INVALID_ARG           # misaligned
    assert call(ws=None) == moe.MOE_ERR_INVALID_ARG
    assert call(ws=FAKE + 16) == moe.MOE_ERR_INVALID_ARG         # workspace not 256-aligned
    assert call(n=n - 1) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert call(d=qwen3(k=0)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    # sigmoid gating needs the selection bias
    d3 = qwen3(T=16, gating=moe.MOE_GATE_SIGMOID_BIAS_RENORM)
    assert lib.moe_route(ctypes.byref(d3), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE,
                         moe.moe_workspace_size(d3), None) == moe.MOE_ERR_INVALID_ARG
    # every argument valid: the call reaches the device check, which fails
    # without a GPU -- there is no host fallback
    assert call() in (moe.MOE_ERR_CUDA, moe.MOE_ERR_UNSUPPORTED_DEVICE)


def test_other_calls_validate(lib):
    d = qwen3(T=16)
    n = moe.moe_workspace_size(d)
    bd = lambda *a: lib.moe_build_dispatch(ctypes.byref(d), *a, FAKE, n, None)
    assert bd(None, None, FAKE, FAKE, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert bd(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE) == moe.MOE_ERR_INVALID_ARG  # w_perm needs topk_w
    ffn = lambda *a: lib.moe_grouped_swiglu_ffn(ctypes.byref(d), *a, FAKE, n, None)
    assert ffn(FAKE, FAKE, FAKE, None, FAKE, None, None, None, FAKE) == moe.MOE_ERR_INVALID_ARG
    ds = qwen3(T=16, shared=True)
    assert lib.moe_grouped_swiglu_ffn(ctypes.byref(ds), FAKE, FAKE, FAKE, None, FAKE, FAKE, None,
                                      None, FAKE, FAKE, moe.moe_workspace_size(ds),
                                      None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(d), FAKE, None, None, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    w = moe.LayerWeights(FAKE, None, FAKE, None, None, None)
    assert lib.moe_layer_forward(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, FAKE, n, None,
                                 None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(None, 256, None) == moe.MOE_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in range(-7, 1):
        s = moe.moe_status_string(code)
        assert s and s != "unknown status"
    assert moe.moe_status_string(-99) == "unknown status"


def test_binding_passes_pointer_width_arguments(lib):
    # Every entry point must be called with pointer-width argument types: a
    # function left with ctypes' default (C int) would truncate device pointers
    # and stream handles.  Calling each Python wrapper with an invalid shape
    # configures its ctypes signature and returns before any launch.
    bad = qwen3(k=0)
    t = FAKE
    for call in (lambda: moe.moe_build_dispatch_noalloc(bad, t, None, t, t, t, t, None, None, t),):
        with pytest.raises(moe.MoeError) as ei:
            call()
        assert ei.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe.h")).read(), flags=re.S)
    for name in declared_functions():
        params = re.search(name + r"\s*\(([^)]*)\)", text).group(1)
        params = [q.strip() for q in params.split(",") if q.strip()]
        f = getattr(lib, name)
        assert f.argtypes is not None, name
        assert len(f.argtypes) == len(params), name
        for decl, a in zip(params, f.argtypes):
            if "*" in decl or decl.startswith("moe_stream_t"):
                assert a is ctypes.c_void_p or issubclass(a, ctypes._Pointer), (name, decl)
            elif decl.startswith("size_t"):
                assert a is ctypes.c_size_t, (name, decl)
            elif decl.startswith("int64_t"):
                assert a is ctypes.c_int64, (name, decl)
            else:
                assert a is ctypes.c_int32, (name, decl)


def test_bounded_wait_check_validates_before_launch(lib):
    # NULL, unaligned or too small workspaces are rejected on the host
    assert lib.moe_check_bounded_wait(None, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_check_bounded_wait(0x10010, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_check_bounded_wait(0x10000, 16, None) == moe.MOE_ERR_INVALID_ARG



def test_forward_path_validation_before_launch(lib):
    w = moe.LayerWeights(FAKE, None, FAKE, FAKE, None, None)
    fwd = lambda d, path: lib.moe_layer_forward_ex(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE,
                                                   FAKE, moe.moe_workspace_size(d), None, None,
                                                   path)
    # an unknown path
    assert fwd(qwen3(T=4), 4) == moe.MOE_ERR_INVALID_ARG
    assert fwd(qwen3(T=4), -1) == moe.MOE_ERR_INVALID_ARG
    # the persistent layer takes at most 16 tokens and H >= 256
    assert fwd(qwen3(T=17), moe.MOE_PATH_PERSISTENT) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert fwd(qwen3(T=4, H=128), moe.MOE_PATH_PERSISTENT) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    # valid otherwise: the device check, which fails without a GPU
    for path in (moe.MOE_PATH_AUTO, moe.MOE_PATH_KERNEL_CHAIN, moe.MOE_PATH_PERSISTENT,
                 moe.MOE_PATH_CHAIN_ONE_SM):
        assert fwd(qwen3(T=4), path) in (moe.MOE_ERR_CUDA, moe.MOE_ERR_UNSUPPORTED_DEVICE)
    assert lib.moe_check_bounded_grid_wait(None, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_check_bounded_grid_wait(0x10000, 16, None) == moe.MOE_ERR_INVALID_ARG


def test_expert_capacity_host_helper(lib):
    import oracle
    for (num, den), T, k, E in [((5, 4), 5, 1, 8), ((1, 1), 16, 1, 8), ((1, 1), 17, 1, 8),
                                ((2, 1), 8192, 8, 128), ((5, 4), 1024, 8, 128),
                                ((3, 7), 33, 4, 16)]:
        assert lib.moe_expert_capacity(num, den, T, k, E) == oracle.expert_capacity(num, den, T * k, E)
    assert lib.moe_expert_capacity(0, 1, 5, 1, 8) == 0
    assert moe.moe_expert_capacity(1.25, 5, 1, 8) == 1
    w = moe.LayerWeights(FAKE, None, FAKE, FAKE, None, None)
    d = qwen3(T=64)
    call = lambda c: lib.moe_layer_forward_capacity(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, c,
                                                     FAKE, moe.moe_workspace_size(d), None)
    assert call(0) == moe.MOE_ERR_INVALID_ARG
    assert call(4) in (moe.MOE_ERR_CUDA, moe.MOE_ERR_UNSUPPORTED_DEVICE)
