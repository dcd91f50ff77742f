"""Python binding of the sm_103a MoE FFN layer library (``libmoe_gb300.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C ABI's names (``include/moe.h``) and take torch
CUDA tensors (or raw device pointers as ints); streams default to torch's
current stream.  There is no CPU fallback: if the library is missing, every
call raises ``LibraryNotBuilt``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_CHECK = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_UNSUPPORTED_DEVICE = -7

MOE_GATE_TOPK_SOFTMAX = 0
MOE_GATE_SOFTMAX_TOPK = 1
MOE_GATE_SOFTMAX_TOPK_RENORM = 2
MOE_GATE_SIGMOID_BIAS_RENORM = 3

MOE_PATH_AUTO = 0
MOE_PATH_KERNEL_CHAIN = 1
MOE_PATH_PERSISTENT = 2
MOE_PATH_CHAIN_ONE_SM = 3

MOE_STAGE_EVENTS = 7
STAGE_NAMES = ("route", "dispatch", "gather", "gateup", "down", "combine")


class LibraryNotBuilt(ImportError):
    pass


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status} ({moe_status_string(status)})")


class LayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("gating", ctypes.c_int32),
                ("has_shared_expert", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("sel_bias", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w13_shared", ctypes.c_void_p), ("w2_shared", ctypes.c_void_p)]


_LAYOUT_FIELDS = ("status", "logits", "topk_ids", "topk_w", "gap", "counts", "offsets",
                  "perm_src", "inv_pos", "w_perm", "x_perm", "h", "out_perm", "plan", "total")


class LayerWeightsFp8(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("sel_bias", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("w13_shared", ctypes.c_void_p), ("w13_shared_scale", ctypes.c_void_p),
                ("w2_shared", ctypes.c_void_p), ("w2_shared_scale", ctypes.c_void_p)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _LAYOUT_FIELDS]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded CUDA library (raises LibraryNotBuilt if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryNotBuilt(f"{LIB_PATH} is missing: build it with "
                              "`python -m routed_expert_ffn_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    D = ctypes.POINTER(LayerDesc)
    sig = {
        "moe_workspace_size": ([D], S),
        "moe_workspace_layout": ([D, ctypes.POINTER(WorkspaceLayout)], I32),
        "moe_workspace_init": ([P, S, P], I32),
        "moe_get_device_status": ([P, S, P, I32, ctypes.POINTER(I32)], I32),
        "moe_status_string": ([I32], ctypes.c_char_p),
        "moe_route": ([D, P, P, P, P, P, P, P, P, S, P], I32),
        "moe_build_dispatch": ([D, P, P, P, P, P, P, P, P, S, P], I32),
        "moe_grouped_swiglu_ffn": ([D, P, P, P, P, P, P, P, P, P, P, S, P], I32),
        "moe_combine": ([D, P, P, P, P, P], I32),
        "moe_layer_forward": ([D, ctypes.POINTER(LayerWeights), P, P, P, S, P, P], I32),
        "moe_check_bounded_wait": ([P, S, P], I32),
        "moe_check_bounded_grid_wait": ([P, S, P], I32),
        "moe_expert_capacity": ([ctypes.c_int64, ctypes.c_int64, I32, I32, I32], I32),
        "moe_quantize_fp8": ([P, I32, I32, I32, P, P, P], I32),
        "moe_layer_forward_fp8": ([D, ctypes.POINTER(LayerWeightsFp8), P, P, P, S, P], I32),
        "moe_layer_forward_capacity": ([D, ctypes.POINTER(LayerWeights), P, P, I32, P, S, P], I32),
        "moe_layer_forward_ex": ([D, ctypes.POINTER(LayerWeights), P, P, P, S, P, P, I32], I32),
        "moe_reshard_ep_to_tp_pack": ([I32, I32, I32, I32, P, P, P, P, P], I32),
        "moe_reshard_tp_to_ep_unpack": ([I32, I32, I32, I32, P, P, P, P, P], I32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


# ---------------------------------------------------------------- helpers --

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != MOE_OK:
        raise MoeError(fn, st)


def desc(T: int, H: int, E: int, k: int, I: int, gating: int, shared: bool = False) -> LayerDesc:
    return LayerDesc(T, H, E, k, I, gating, 1 if shared else 0)


# ---------------------------------------------------------------- host API --

def moe_status_string(status: int) -> str:
    return library().moe_status_string(status).decode()


def moe_workspace_size(d: LayerDesc) -> int:
    return int(library().moe_workspace_size(ctypes.byref(d)))


def moe_workspace_layout(d: LayerDesc) -> Dict[str, int]:
    out = WorkspaceLayout()
    _check("moe_workspace_layout", library().moe_workspace_layout(ctypes.byref(d), ctypes.byref(out)))
    return {n: int(getattr(out, n)) for n in _LAYOUT_FIELDS}


def alloc_workspace(d: LayerDesc, device="cuda"):
    """A zero-initialised workspace tensor (uint8) of moe_workspace_size(d) bytes."""
    import torch
    n = moe_workspace_size(d)
    if n == 0:
        raise MoeError("moe_workspace_size", MOE_ERR_UNSUPPORTED_SHAPE)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_workspace_init(ws, stream=None):
    _check("moe_workspace_init", library().moe_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)))


def moe_get_device_status(ws, clear: bool = True, stream=None):
    """(status, raw bits) of the workspace's device status word (synchronises)."""
    raw = ctypes.c_int32(0)
    st = library().moe_get_device_status(_ptr(ws), _nbytes(ws), _stream(stream), 1 if clear else 0,
                                         ctypes.byref(raw))
    return int(st), int(raw.value)


def moe_check_bounded_grid_wait(ws, stream=None):
    """Launch the grid-barrier wait check (about one second on the GPU); read the
    result with moe_get_device_status (MOE_ERR_TIMEOUT, bit 7), then call
    moe_workspace_init."""
    _check("moe_check_bounded_grid_wait",
           library().moe_check_bounded_grid_wait(_ptr(ws), _nbytes(ws), _stream(stream)))


def moe_check_bounded_wait(ws, stream=None):
    """Launch the bounded-wait check (about one second on the GPU); read the
    result with moe_get_device_status (MOE_ERR_TIMEOUT, bit 6)."""
    _check("moe_check_bounded_wait",
           library().moe_check_bounded_wait(_ptr(ws), _nbytes(ws), _stream(stream)))


# ------------------------------------------------------------- compute API --

def moe_route(d: LayerDesc, x, w_router, sel_bias, logits, topk_ids, topk_w, boundary_gap, ws,
              stream=None):
    _check("moe_route", library().moe_route(
        ctypes.byref(d), _ptr(x), _ptr(w_router), _ptr(sel_bias), _ptr(logits), _ptr(topk_ids),
        _ptr(topk_w), _ptr(boundary_gap), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_build_dispatch(d: LayerDesc, topk_ids, topk_w, counts, offsets, perm_src, inv_pos, w_perm,
                       ws, stream=None):
    _check("moe_build_dispatch", library().moe_build_dispatch(
        ctypes.byref(d), _ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm_src),
        _ptr(inv_pos), _ptr(w_perm), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_grouped_swiglu_ffn(d: LayerDesc, x, perm_src, offsets, w_perm, w13, w2, w13_shared,
                           w2_shared, out_perm, ws, stream=None):
    _check("moe_grouped_swiglu_ffn", library().moe_grouped_swiglu_ffn(
        ctypes.byref(d), _ptr(x), _ptr(perm_src), _ptr(offsets), _ptr(w_perm), _ptr(w13), _ptr(w2),
        _ptr(w13_shared), _ptr(w2_shared), _ptr(out_perm), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_combine(d: LayerDesc, out_perm, inv_pos, topk_w, y, stream=None):
    _check("moe_combine", library().moe_combine(
        ctypes.byref(d), _ptr(out_perm), _ptr(inv_pos), _ptr(topk_w), _ptr(y), _stream(stream)))


def moe_reshard_ep_to_tp_pack(E_local: int, H: int, I: int, P: int, w13, w2, w13_chunks,
                              w2_chunks, stream=None):
    """EP -> TP local permute: [E_l,2I,H] / [E_l,H,I] -> per-peer chunks
    [P,E_l,2I/P,H] / [P,E_l,H,I/P] (either pair may be None)."""
    _check("moe_reshard_ep_to_tp_pack", library().moe_reshard_ep_to_tp_pack(
        E_local, H, I, P, _ptr(w13), _ptr(w2), _ptr(w13_chunks), _ptr(w2_chunks),
        _stream(stream)))


def moe_reshard_tp_to_ep_unpack(E_local: int, H: int, I: int, P: int, w13_chunks, w2_chunks, w13,
                                w2, stream=None):
    """TP -> EP local permute, the inverse of moe_reshard_ep_to_tp_pack."""
    _check("moe_reshard_tp_to_ep_unpack", library().moe_reshard_tp_to_ep_unpack(
        E_local, H, I, P, _ptr(w13_chunks), _ptr(w2_chunks), _ptr(w13), _ptr(w2),
        _stream(stream)))


def layer_weights(w_router, w13, w2, sel_bias=None, w13_shared=None, w2_shared=None) -> LayerWeights:
    return LayerWeights(_ptr(w_router), _ptr(sel_bias), _ptr(w13), _ptr(w2), _ptr(w13_shared),
                        _ptr(w2_shared))


def moe_layer_forward(d: LayerDesc, w: LayerWeights, x, y, ws, stream=None,
                      stage_events: Optional[Sequence] = None, path: int = None):
    """Whole layer forward.  ``stage_events``: None or MOE_STAGE_EVENTS torch.cuda.Event
    objects (created with enable_timing and already recorded once) or raw handles.
    ``path``: None (moe_layer_forward, automatic choice) or one of MOE_PATH_*
    (moe_layer_forward_ex)."""
    ev = None
    if stage_events is not None:
        if len(stage_events) != MOE_STAGE_EVENTS:
            raise ValueError(f"need {MOE_STAGE_EVENTS} events")
        ev = (ctypes.c_void_p * MOE_STAGE_EVENTS)(
            *[e if isinstance(e, int) else e.cuda_event for e in stage_events])
    if path is None:
        _check("moe_layer_forward", library().moe_layer_forward(
            ctypes.byref(d), ctypes.byref(w), _ptr(x), _ptr(y), _ptr(ws), _nbytes(ws),
            _stream(stream), ev))
    else:
        _check("moe_layer_forward_ex", library().moe_layer_forward_ex(
            ctypes.byref(d), ctypes.byref(w), _ptr(x), _ptr(y), _ptr(ws), _nbytes(ws),
            _stream(stream), ev, int(path)))


def moe_expert_capacity(cf, T: int, k: int, E: int) -> int:
    """C = ceil(cf * T * k / E); cf a Fraction, an int, or a float (taken as the
    nearest fraction with a denominator up to 10^6)."""
    from fractions import Fraction
    f = Fraction(cf).limit_denominator(10 ** 6)
    c = library().moe_expert_capacity(f.numerator, f.denominator, T, k, E)
    if c <= 0:
        raise ValueError("invalid capacity factor or shape")
    return int(c)


def moe_layer_forward_capacity(d: LayerDesc, w: LayerWeights, x, y, capacity: int, ws,
                               stream=None):
    """Layer forward with at most ``capacity`` assignments per routed expert
    (the first ones in token order; the rest dropped)."""
    _check("moe_layer_forward_capacity", library().moe_layer_forward_capacity(
        ctypes.byref(d), ctypes.byref(w), _ptr(x), _ptr(y), int(capacity), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def moe_quantize_fp8(w, n: int, rows: int, K: int, q, scale_exp, stream=None):
    """E4M3 codes q [n,rows,K] (uint8) and block exponents scale_exp
    [n, ceil(rows/128), ceil(K/128)] (int8) of bf16 matrices w [n,rows,K]."""
    _check("moe_quantize_fp8", library().moe_quantize_fp8(
        _ptr(w), int(n), int(rows), int(K), _ptr(q), _ptr(scale_exp), _stream(stream)))


def quantize_layer_fp8(w13, w2, w13_shared=None, w2_shared=None):
    """Device tensors (codes and block exponents) of a layer's expert weights:
    w13 [E,2I,H] and w2 [E,H,I] bf16 (and the shared expert's)."""
    import torch
    out = {}

    def q(name, w, n, rows, K, lead):
        codes = torch.empty(tuple(w.shape), dtype=torch.uint8, device=w.device)
        sc = torch.empty(lead + (-(-rows // 128), -(-K // 128)), dtype=torch.int8,
                         device=w.device)
        moe_quantize_fp8(w, n, rows, K, codes, sc)
        out[name] = codes
        out[name + "_scale"] = sc

    E, I2, H = w13.shape
    q("w13", w13, 2 * E, I2 // 2, H, (E, 2))      # [E,2,ceil(I/128),ceil(H/128)]
    q("w2", w2, E, H, I2 // 2, (E,))              # [E,ceil(H/128),ceil(I/128)]
    if w13_shared is not None:
        q("w13_shared", w13_shared, 2, I2 // 2, H, (2,))
        q("w2_shared", w2_shared, 1, H, I2 // 2, ())
    return out


def layer_weights_fp8(w_router, q: Dict, sel_bias=None) -> LayerWeightsFp8:
    """The C struct over quantised expert weights (quantize_layer_fp8's dict)."""
    g = lambda k: _ptr(q.get(k))
    return LayerWeightsFp8(_ptr(w_router), _ptr(sel_bias), g("w13"), g("w13_scale"), g("w2"),
                           g("w2_scale"), g("w13_shared"), g("w13_shared_scale"), g("w2_shared"),
                           g("w2_shared_scale"))


def moe_layer_forward_fp8(d: LayerDesc, w: LayerWeightsFp8, x, y, ws, stream=None):
    """Layer forward with FP8 expert weights: the persistent decode layer up to
    16 tokens, else the kernel chain with FP8 GEMMs on fp16 token rows."""
    _check("moe_layer_forward_fp8", library().moe_layer_forward_fp8(
        ctypes.byref(d), ctypes.byref(w), _ptr(x), _ptr(y), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def workspace_view(ws, layout: Dict[str, int], name: str, dtype, shape):
    """A tensor view of one buffer moe_layer_forward leaves in the workspace."""
    import torch
    itemsize = torch.empty((), dtype=dtype).element_size()
    n = 1
    for s in shape:
        n *= s
    off = layout[name]
    return ws[off:off + n * itemsize].view(dtype).view(*shape)


def moe_build_dispatch_noalloc(d: LayerDesc, topk_ids, topk_w, counts, offsets, perm_src, inv_pos,
                               w_perm, device_status=None, stream=None):
    """moe_build_dispatch without a workspace, for callers that cannot allocate
    device memory: the dispatch scratch lives in a fixed array inside the
    library (MOE_NOALLOC_SCRATCH_BYTES, held until the process exits).  Calls
    share that array, so calls that overlap on the GPU race; order them on one
    stream.  Too large a batch raises MoeError(MOE_ERR_UNSUPPORTED_SHAPE)."""
    f = library().moe_build_dispatch_noalloc
    if f.argtypes is None:
        # pointer-width arguments: without argtypes ctypes would pass ints as C int
        P = ctypes.c_void_p
        f.argtypes = [ctypes.POINTER(LayerDesc), P, P, P, P, P, P, P, P, P]
        f.restype = ctypes.c_int32
    _check("moe_build_dispatch_noalloc", f(
        ctypes.byref(d), _ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm_src),
        _ptr(inv_pos), _ptr(w_perm), _ptr(device_status), _stream(stream)))
