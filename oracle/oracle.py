"""ctypes front end of the CPU oracle (moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the bench's CPU-baseline leg may
import this module; the product package never does.  It builds the oracle with the
host C++ compiler into oracle/_build/ (plain -O2, FP contraction off so x86 and Arm
hosts round identically) and exposes numpy-level wrappers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or older than its sources."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fPIC", "-shared",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_e2m1_value.restype = ctypes.c_float
            L.oracle_e2m1_value.argtypes = [ctypes.c_uint32]
            L.oracle_e4m3_value.restype = ctypes.c_float
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint32]
            L.oracle_dequant_row.argtypes = [_P, _P, ctypes.c_float, ctypes.c_int, _P]
            for name in ("oracle_route_topk_f32", "oracle_route_topk_f64"):
                getattr(L, name).argtypes = [ctypes.c_int] * 3 + [_P] * 3
            L.oracle_plan.argtypes = [ctypes.c_int] * 3 + [_P] * 4
            for name in ("oracle_moe_experts_f32", "oracle_moe_experts_f64"):
                getattr(L, name).argtypes = ([ctypes.c_int] * 5 + [_P] * 5 + [ctypes.c_float]
                                             + [_P] * 2 + [ctypes.c_float] + [_P] * 3)
            L.oracle_moe_experts_ts_f32.argtypes = [ctypes.c_int] * 5 + [_P] * 12
            L.oracle_bf16_round.restype = ctypes.c_uint16
            L.oracle_bf16_round.argtypes = [ctypes.c_float]
            for name in ("oracle_router_logits_f32", "oracle_router_logits_f64"):
                getattr(L, name).argtypes = [ctypes.c_int] * 3 + [_P] * 3
            for name in ("oracle_gated_residual_norm_f32", "oracle_gated_residual_norm_f64"):
                getattr(L, name).argtypes = [ctypes.c_int] * 3 + [_P] * 4 + [ctypes.c_float] + [_P] * 2
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def e2m1_value(nibble: int) -> float:
    return float(lib().oracle_e2m1_value(int(nibble)))


def e4m3_value(byte: int) -> float:
    return float(lib().oracle_e4m3_value(int(byte)))


def dequant_row(codes: np.ndarray, scales: np.ndarray, tensor_scale: float, K: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    assert codes.size == K // 2 and scales.size == K // 16
    out = np.empty(K, dtype=np.float32)
    rc = lib().oracle_dequant_row(_ptr(codes), _ptr(scales), float(tensor_scale), K, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dequant_row: invalid arguments")
    return out


def route_topk(logits: np.ndarray, k: int, precision: str = "f32"):
    """ids int32 [T,k] and weights [T,k] (float32 or float64) of the oracle router."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    if precision == "f32":
        w = np.empty((T, k), dtype=np.float32)
        rc = lib().oracle_route_topk_f32(T, E, k, _ptr(logits), _ptr(ids), _ptr(w))
    elif precision == "f64":
        w = np.empty((T, k), dtype=np.float64)
        rc = lib().oracle_route_topk_f64(T, E, k, _ptr(logits), _ptr(ids), _ptr(w))
    else:
        raise ValueError(precision)
    if rc != 0:
        raise ValueError("oracle_route_topk: invalid arguments")
    return ids, w


def plan(ids: np.ndarray, E: int):
    """counts [E], offsets [E+1], touched [U] of the oracle bucketing."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    touched = np.empty(E, dtype=np.int32)
    U = lib().oracle_plan(T, E, k, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(touched))
    if U < 0:
        raise ValueError("oracle_plan: invalid ids")
    return counts, offsets, touched[:U].copy()


def moe_experts(dims, hidden_bf16: np.ndarray, ids: np.ndarray, weights: np.ndarray, w: dict,
                residual_bf16: np.ndarray | None = None, token_mask: np.ndarray | None = None,
                precision: str = "f32", out: np.ndarray | None = None) -> np.ndarray:
    """Expert FFN + weighted un-route + residual for the masked tokens.

    dims = (T, d, F, E, k).  Returns out [T, d] in the oracle's precision; rows of
    unmasked tokens are NaN (or whatever `out` held)."""
    T, d, F, E, k = (int(v) for v in dims)
    dt = np.float32 if precision == "f32" else np.float64
    hidden_bf16 = np.ascontiguousarray(hidden_bf16, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=dt)
    arrs = [np.ascontiguousarray(w[n], dtype=np.uint8) for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")]
    res = None if residual_bf16 is None else np.ascontiguousarray(residual_bf16, dtype=np.uint16)
    mask = None if token_mask is None else np.ascontiguousarray(token_mask, dtype=np.uint8)
    if out is None:
        out = np.full((T, d), np.nan, dtype=dt)
    fn = lib().oracle_moe_experts_f32 if precision == "f32" else lib().oracle_moe_experts_f64
    rc = fn(T, d, F, E, k, _ptr(hidden_bf16), _ptr(ids), _ptr(weights),
            _ptr(arrs[0]), _ptr(arrs[1]), float(w["w13_ts"]), _ptr(arrs[2]), _ptr(arrs[3]),
            float(w["w2_ts"]), 0 if res is None else _ptr(res), 0 if mask is None else _ptr(mask),
            _ptr(out))
    if rc != 0:
        raise ValueError("oracle_moe_experts: invalid arguments")
    return out


def moe_layer(cfg, inputs: dict, token_mask=None, precision: str = "f32"):
    """Router + experts of one layer call on moe_inputs-style inputs.

    Returns (ids, weights, out)."""
    ids, wts = route_topk(inputs["logits"], cfg.k, precision)
    out = moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inputs["hidden"], ids, wts, inputs,
                      inputs.get("residual"), token_mask, precision)
    return ids, wts, out


def bf16_round(x) -> np.ndarray:
    """BF16 bit patterns (uint16) of float32 values, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    f = lib().oracle_bf16_round
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def router_logits(hidden_bf16: np.ndarray, router_w_bf16: np.ndarray, precision: str = "f32") -> np.ndarray:
    """logits [T, E] = hidden [T, d] (BF16 bits) x router_w [E, d] (BF16 bits)^T."""
    hidden_bf16 = np.ascontiguousarray(hidden_bf16, dtype=np.uint16)
    router_w_bf16 = np.ascontiguousarray(router_w_bf16, dtype=np.uint16)
    T, d = hidden_bf16.shape
    E, d2 = router_w_bf16.shape
    assert d == d2
    dt = np.float32 if precision == "f32" else np.float64
    out = np.empty((T, E), dtype=dt)
    fn = lib().oracle_router_logits_f32 if precision == "f32" else lib().oracle_router_logits_f64
    if fn(T, d, E, _ptr(hidden_bf16), _ptr(router_w_bf16), _ptr(out)) != 0:
        raise ValueError("oracle_router_logits: invalid arguments")
    return out


def gated_residual_norm(moe_out: np.ndarray, residual_bf16: np.ndarray, inject_logits: np.ndarray,
                        norm_w_bf16: np.ndarray, eps: float = 1e-6, precision: str = "f32"):
    """(R' [G, T, d] BF16 bits, N [G, T, d]) of the gated residual update and GemmaRMSNorm."""
    dt = np.float32 if precision == "f32" else np.float64
    moe_out = np.ascontiguousarray(moe_out, dtype=dt)
    residual_bf16 = np.ascontiguousarray(residual_bf16, dtype=np.uint16)
    inject_logits = np.ascontiguousarray(inject_logits, dtype=np.float32)
    norm_w_bf16 = np.ascontiguousarray(norm_w_bf16, dtype=np.uint16)
    G, T, d = residual_bf16.shape
    assert moe_out.shape == (T, d) and inject_logits.shape == (T, G) and norm_w_bf16.shape == (G, d)
    r_out = np.empty((G, T, d), dtype=np.uint16)
    n_out = np.empty((G, T, d), dtype=dt)
    fn = lib().oracle_gated_residual_norm_f32 if precision == "f32" else lib().oracle_gated_residual_norm_f64
    if fn(T, d, G, _ptr(moe_out), _ptr(residual_bf16), _ptr(inject_logits), _ptr(norm_w_bf16), float(eps),
          _ptr(r_out), _ptr(n_out)) != 0:
        raise ValueError("oracle_gated_residual_norm: invalid arguments")
    return r_out, n_out


def moe_experts_ts(dims, hidden_bf16, ids, weights, w: dict, w13_ts_e, w2_ts_e, residual_bf16=None,
                   token_mask=None) -> np.ndarray:
    """oracle moe_experts (FP32) with per-expert tensor scales w13_ts_e [E], w2_ts_e [E]."""
    T, d, F, E, k = (int(v) for v in dims)
    hidden_bf16 = np.ascontiguousarray(hidden_bf16, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    arrs = [np.ascontiguousarray(w[n], dtype=np.uint8) for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")]
    t13 = np.ascontiguousarray(w13_ts_e, dtype=np.float32)
    t2 = np.ascontiguousarray(w2_ts_e, dtype=np.float32)
    assert t13.shape == (E,) and t2.shape == (E,)
    res = None if residual_bf16 is None else np.ascontiguousarray(residual_bf16, dtype=np.uint16)
    mask = None if token_mask is None else np.ascontiguousarray(token_mask, dtype=np.uint8)
    out = np.full((T, d), np.nan, dtype=np.float32)
    rc = lib().oracle_moe_experts_ts_f32(T, d, F, E, k, _ptr(hidden_bf16), _ptr(ids), _ptr(weights), _ptr(arrs[0]),
                                         _ptr(arrs[1]), _ptr(t13), _ptr(arrs[2]), _ptr(arrs[3]), _ptr(t2),
                                         0 if res is None else _ptr(res), 0 if mask is None else _ptr(mask),
                                         _ptr(out))
    if rc != 0:
        raise ValueError("oracle_moe_experts_ts: invalid arguments")
    return out
