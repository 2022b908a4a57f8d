"""ctypes binding of libroutedmoe.so: argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module turns torch
tensors into device pointers and the current torch stream into a cudaStream_t.  If the
shared library has not been built, every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libroutedmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE = -5

MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_TIMEOUT = 0x2
MOE_DEV_HIDDEN_RANGE = 0x4
MOE_DEV_H_SATURATED = 0x8
MOE_DEV_Y_SATURATED = 0x10

ALGO_AUTO = 0
ALGO_TCGEN05 = 1
ALGO_SIMT = 2
ALGO_MMA = 3
ALGO_WIDE = 4

# Every function declared in include/moe.h, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


_SP = ctypes.POINTER(Shape)
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "moe_workspace_init": (_I, [_P, ctypes.c_size_t, _P]),
    "moe_check_shape": (_I, [_SP]),
    "moe_auto_algo": (_I, [_SP]),
    "moe_layer_launches": (_I, [_SP]),
    "moe_static_workspace_read_status": (_I, [_I, ctypes.POINTER(ctypes.c_uint32), _P]),
    "moe_unroute_fused": (_I, [_SP, _I]),
    "moe_route_topk": (_I, [_SP, _P, _P, _P, _P]),
    "moe_plan": (_I, [_SP, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward": (_I, [_SP, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_algo": (_I, [_SP, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _I, _P]),
    "moe_forward_prepare": (_I, [_SP, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_experts": (_I, [_SP, _P, _P, _F, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _I, _P]),
    "moe_forward_expert_kernels": (_I, [_SP, _P, _P, _F, _P, _P, _F, _P, ctypes.c_size_t, _I, _P]),
    "moe_forward_unroute": (_I, [_SP, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_front": (_I, [_SP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_layer": (_I, [_SP, _P, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_layer_expert_range": (_I, [_SP, _I, _I, _P, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, _P, _P,
                                    ctypes.c_size_t, _P]),
    "moe_plan_expert_range": (_I, [_SP, _I, _I, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_experts_expert_range": (_I, [_SP, _I, _I, _P, _P, _F, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _I,
                                              _P]),
    "moe_layer_expert_scales": (_I, [_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_router_logits": (_I, [_SP, _P, _P, _P, _P]),
    "moe_layer_from_hidden": (_I, [_SP, _P, _P, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_forward_unroute_gated": (_I, [_SP, _I, _P, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_layer_gated": (_I, [_SP, _I, _P, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, _F, _P, _P, _P, _P, _P,
                             ctypes.c_size_t, _P]),
    "moe_layer_static_workspace": (_I, [_SP, _P, _P, _P, _P, _F, _P, _P, _F, _P, _P, _P, _P, _P]),
    "moe_read_device_status": (_I, [_P, _I, ctypes.POINTER(ctypes.c_uint32), _P]),
    "moe_plan_summary": (_I, [_SP, _P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_plan_views": (_I, [_SP, _P] + [ctypes.POINTER(ctypes.c_void_p)] * 5),
    # include/moe_selftest.h
    "moe_selftest_expert_timeout": (_I, [_SP, _P, _P, _F, _P, _P, _F, _P, _P, _P, ctypes.c_size_t, _I, _I,
                                         ctypes.c_longlong, _P]),
    "moe_selftest_expert_part": (_I, [_SP, _P, _P, _F, _P, _P, _F, _P, ctypes.c_size_t, _I, _I, _P]),
}

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn, rc):
        msg = lib().moe_status_string(rc).decode()
        extra = lib().moe_last_cuda_error().decode()
        show = extra and rc in (MOE_ERR_CUDA, MOE_ERR_WORKSPACE)
        super().__init__(f"{fn} -> {rc} ({msg}){': ' + extra if show else ''}")
        self.rc = rc


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA extension first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def shape_of(T, d, ffn, E, k) -> Shape:
    return Shape(int(T), int(d), int(ffn), int(E), int(k))


def workspace_bytes(shape: Shape) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(shape)))


def check_shape(shape: Shape) -> int:
    return int(lib().moe_check_shape(ctypes.byref(shape)))


def unroute_fused(shape: Shape, algo: int = ALGO_AUTO) -> bool:
    """True if the expert kernel of `algo` runs the un-route itself for `shape`."""
    rc = int(lib().moe_unroute_fused(ctypes.byref(shape), int(algo)))
    if rc < 0:
        raise MoeError("moe_unroute_fused", rc)
    return rc == 1


def layer_launches(shape: Shape) -> int:
    """Kernel launches of one moe_layer call for `shape` (1: the one-launch layer)."""
    rc = int(lib().moe_layer_launches(ctypes.byref(shape)))
    if rc < 0:
        raise MoeError("moe_layer_launches", rc)
    return rc


def auto_algo(shape: Shape) -> int:
    """The expert kernel ALGO_AUTO picks for `shape` (ALGO_MMA or ALGO_TCGEN05)."""
    rc = int(lib().moe_auto_algo(ctypes.byref(shape)))
    if rc < 0:
        raise MoeError("moe_auto_algo", rc)
    return rc


class Workspace:
    """Caller-owned device workspace for one shape (allocated through torch)."""

    def __init__(self, shape: Shape, device="cuda", stream=None):
        self.shape = shape
        self.nbytes = workspace_bytes(shape)
        if self.nbytes == 0:
            raise MoeError("moe_workspace_bytes", MOE_ERR_UNSUPPORTED)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.tensor = self.buf[off:off + self.nbytes]
        _check("moe_workspace_init", lib().moe_workspace_init(_ptr(self.tensor), self.nbytes, _stream(stream)))

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())


def route_topk(shape: Shape, logits, ids, weights, stream=None):
    _check("moe_route_topk", lib().moe_route_topk(ctypes.byref(shape), _ptr(logits), _ptr(ids), _ptr(weights),
                                                  _stream(stream)))


def plan(shape: Shape, ids, weights, ws: Workspace, stream=None):
    _check("moe_plan", lib().moe_plan(ctypes.byref(shape), _ptr(ids), _ptr(weights), ws.ptr, ws.nbytes,
                                      _stream(stream)))


def forward(shape: Shape, hidden, w: dict, residual, out, ws: Workspace, algo: int = ALGO_AUTO, stream=None):
    _check("moe_forward_algo", lib().moe_forward_algo(
        ctypes.byref(shape), _ptr(hidden), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), float(w["w13_ts"]),
        _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual), _ptr(out), ws.ptr,
        ws.nbytes, int(algo), _stream(stream)))


def forward_prepare(shape: Shape, hidden, ws: Workspace, stream=None):
    _check("moe_forward_prepare", lib().moe_forward_prepare(ctypes.byref(shape), _ptr(hidden), ws.ptr, ws.nbytes,
                                                            _stream(stream)))


def forward_experts(shape: Shape, w: dict, residual, out, ws: Workspace, algo: int = ALGO_AUTO, stream=None):
    _check("moe_forward_experts", lib().moe_forward_experts(
        ctypes.byref(shape), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), float(w["w13_ts"]),
        _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual), _ptr(out), ws.ptr,
        ws.nbytes, int(algo), _stream(stream)))


def forward_expert_kernels(shape: Shape, w: dict, ws: Workspace, algo: int = ALGO_AUTO, stream=None):
    """The expert kernel(s) alone (per-route down outputs into the workspace)."""
    _check("moe_forward_expert_kernels", lib().moe_forward_expert_kernels(
        ctypes.byref(shape), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), float(w["w13_ts"]),
        _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), ws.ptr, ws.nbytes, algo, _stream(stream)))


def selftest_expert_part(shape: Shape, w: dict, ws: Workspace, algo: int, part: int, stream=None):
    """moe_forward_expert_kernels in two parts (include/moe_selftest.h): part 0 the kernels that
    prepare the expert kernel's input (wide path only), part 1 the expert kernel alone."""
    _check("moe_selftest_expert_part", lib().moe_selftest_expert_part(
        ctypes.byref(shape), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), float(w["w13_ts"]),
        _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), ws.ptr, ws.nbytes, int(algo), int(part),
        _stream(stream)))


def forward_unroute(shape: Shape, residual, out, ws: Workspace, stream=None):
    """The weighted un-route alone: out = residual + the token's routes in slot order."""
    _check("moe_forward_unroute", lib().moe_forward_unroute(
        ctypes.byref(shape), _ptr(residual), _ptr(out), ws.ptr, ws.nbytes, _stream(stream)))


def front(shape: Shape, logits, hidden, ids, weights, ws: Workspace, stream=None):
    _check("moe_front", lib().moe_front(ctypes.byref(shape), _ptr(logits), _ptr(hidden), _ptr(ids), _ptr(weights),
                                        ws.ptr, ws.nbytes, _stream(stream)))


def layer(shape: Shape, logits, hidden, w: dict, residual, out, ids, weights, ws: Workspace, stream=None):
    _check("moe_layer", lib().moe_layer(
        ctypes.byref(shape), _ptr(logits), _ptr(hidden), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]),
        float(w["w13_ts"]), _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual),
        _ptr(out), _ptr(ids), _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def layer_expert_range(shape: Shape, e_begin: int, e_end: int, logits, hidden, w: dict, residual, out, ids,
                       weights, ws: Workspace, stream=None):
    """moe_layer restricted to the experts [e_begin, e_end) (one expert-parallel shard); `w`
    holds those experts' weights only (entry e - e_begin is expert e)."""
    _check("moe_layer_expert_range", lib().moe_layer_expert_range(
        ctypes.byref(shape), int(e_begin), int(e_end), _ptr(logits), _ptr(hidden), _ptr(w["w13_codes"]),
        _ptr(w["w13_scales"]), float(w["w13_ts"]), _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]),
        _ptr(residual), _ptr(out), _ptr(ids), _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def plan_expert_range(shape: Shape, e_begin: int, e_end: int, ids, weights, ws: Workspace, stream=None):
    """moe_plan restricted to the experts [e_begin, e_end) (one expert-parallel shard)."""
    _check("moe_plan_expert_range", lib().moe_plan_expert_range(
        ctypes.byref(shape), int(e_begin), int(e_end), _ptr(ids), _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def forward_experts_expert_range(shape: Shape, e_begin: int, e_end: int, w: dict, residual, out, ws: Workspace,
                                 algo: int = ALGO_AUTO, stream=None):
    """moe_forward_experts on a plan of moe_plan_expert_range with the same range; `w` holds
    the local experts' weights only (entry e - e_begin is expert e)."""
    _check("moe_forward_experts_expert_range", lib().moe_forward_experts_expert_range(
        ctypes.byref(shape), int(e_begin), int(e_end), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]),
        float(w["w13_ts"]), _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual), _ptr(out),
        ws.ptr, ws.nbytes, int(algo), _stream(stream)))


def selftest_expert_timeout(shape: Shape, w: dict, residual, out, ws: Workspace, algo: int, dn_task: int,
                            wait_limit_cycles: int, stream=None):
    """Run the expert kernel on the plan in `ws` with one down task made to wait for a readiness
    counter nobody publishes and every wait limited to `wait_limit_cycles` (include/moe_selftest.h)."""
    _check("moe_selftest_expert_timeout", lib().moe_selftest_expert_timeout(
        ctypes.byref(shape), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), float(w["w13_ts"]), _ptr(w["w2_codes"]),
        _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual), _ptr(out), ws.ptr, ws.nbytes, int(algo),
        int(dn_task), int(wait_limit_cycles), _stream(stream)))


def layer_expert_scales(shape: Shape, logits, hidden, w: dict, w13_ts_e, w2_ts_e, residual, out, ids, weights,
                        ws: Workspace, stream=None):
    """moe_layer with per-expert FP32 tensor scales (device tensors [E]) for W13 and W2."""
    _check("moe_layer_expert_scales", lib().moe_layer_expert_scales(
        ctypes.byref(shape), _ptr(logits), _ptr(hidden), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]), _ptr(w13_ts_e),
        _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), _ptr(w2_ts_e), _ptr(residual), _ptr(out), _ptr(ids),
        _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def router_logits(shape: Shape, hidden, router_w, logits, stream=None):
    """logits [T, E] FP32 = hidden [T, d] BF16 x router_w [E, d] BF16^T (weight-prefetch GEMV)."""
    _check("moe_router_logits", lib().moe_router_logits(ctypes.byref(shape), _ptr(hidden), _ptr(router_w),
                                                        _ptr(logits), _stream(stream)))


def layer_from_hidden(shape: Shape, hidden, router_w, logits, w: dict, residual, out, ids, weights, ws: Workspace,
                      stream=None):
    """The router projection into `logits`, then the whole layer on them (moe_layer)."""
    _check("moe_layer_from_hidden", lib().moe_layer_from_hidden(
        ctypes.byref(shape), _ptr(hidden), _ptr(router_w), _ptr(logits), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]),
        float(w["w13_ts"]), _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual), _ptr(out),
        _ptr(ids), _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def forward_unroute_gated(shape: Shape, G: int, residual, inject_logits, norm_weight, eps: float, residual_out,
                          normed_out, ws: Workspace, stream=None):
    """Gated residual update of G branches plus GemmaRMSNorm from the per-route outputs in `ws`."""
    _check("moe_forward_unroute_gated", lib().moe_forward_unroute_gated(
        ctypes.byref(shape), int(G), _ptr(residual), _ptr(inject_logits), _ptr(norm_weight), float(eps),
        _ptr(residual_out), _ptr(normed_out), ws.ptr, ws.nbytes, _stream(stream)))


def layer_gated(shape: Shape, G: int, logits, hidden, w: dict, residual, inject_logits, norm_weight, eps: float,
                residual_out, normed_out, ids, weights, ws: Workspace, stream=None):
    """Whole layer with the gated residual update and GemmaRMSNorm in place of the plain un-route."""
    _check("moe_layer_gated", lib().moe_layer_gated(
        ctypes.byref(shape), int(G), _ptr(logits), _ptr(hidden), _ptr(w["w13_codes"]), _ptr(w["w13_scales"]),
        float(w["w13_ts"]), _ptr(w["w2_codes"]), _ptr(w["w2_scales"]), float(w["w2_ts"]), _ptr(residual),
        _ptr(inject_logits), _ptr(norm_weight), float(eps), _ptr(residual_out), _ptr(normed_out), _ptr(ids),
        _ptr(weights), ws.ptr, ws.nbytes, _stream(stream)))


def read_status(ws: Workspace, clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    rc = lib().moe_read_device_status(ws.ptr, 1 if clear else 0, ctypes.byref(bits), _stream(stream))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoeError("moe_read_device_status", rc)
    return int(bits.value)


def plan_summary(shape: Shape, ws: Workspace, stream=None):
    u = ctypes.c_int32(0)
    m = ctypes.c_int32(0)
    _check("moe_plan_summary", lib().moe_plan_summary(ctypes.byref(shape), ws.ptr, ctypes.byref(u),
                                                      ctypes.byref(m), _stream(stream)))
    return int(u.value), int(m.value)


def plan_views(shape: Shape, ws: Workspace):
    """Device tensors viewing the plan arrays inside the workspace."""
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    _check("moe_plan_views", lib().moe_plan_views(ctypes.byref(shape), ws.ptr, *[ctypes.byref(p) for p in ptrs]))
    base = ws.tensor.data_ptr()
    R = shape.T * shape.k
    sizes = [shape.E, shape.E + 1, shape.E, R, R]
    out = []
    for p, n in zip(ptrs, sizes):
        off = p.value - base
        out.append(ws.tensor[off:off + 4 * n].view(torch.int32))
    return dict(zip(("counts", "offsets", "touched", "route_pos", "pos_token"), out))
