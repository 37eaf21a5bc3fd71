"""CPU fp64 oracle of the MoE FFN layer with SelectedSoftmax routing.

TEST INFRASTRUCTURE ONLY.  Imported by tests/, by the smoke check and by the
benchmark's CPU-baseline / reference leg; never by the CUDA product path.  The
arithmetic lives in moe_oracle.c (plain C, fp64); this module compiles it with
gcc and marshals numpy arrays through ctypes.

parity: pinned by tests/test_oracle.py against invariants of the definition
("New Community Model: ZONOS3-Mini (Zyphra) - #1271", §Framework change),
closed forms, a hand-derived worked example and a dense numpy brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

F32, BF16, Q8_0 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so beside it (gcc, -O2)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts agree bit for bit.
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        lib.oracle_default_threads.restype = i
        lib.oracle_router_logits.argtypes = [vp, i, i, i, vp, i, dp, i]
        lib.oracle_selected_softmax.argtypes = [dp, vp, i, i, i, vp, dp, dp]
        lib.oracle_softmax_of_set.argtypes = [dp, i, i, i, vp, dp]
        lib.oracle_permute.argtypes = [vp, i, i, i, vp, vp, vp, vp]
        lib.oracle_expert_combine.argtypes = [vp, i, i, i, vp, dp, i, vp, vp, vp, i, i, i, dp, i]
        lib.oracle_moe_forward.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, dp,
                                           vp, dp, dp, i]
        lib.oracle_route_scored.argtypes = [dp, vp, i, i, i, i, vp, dp, dp]
        lib.oracle_moe_forward_scored.argtypes = [vp, i, i, i, vp, vp, i, i, i, vp, vp, vp, i, i,
                                                  dp, vp, dp, dp, i]
        for name in ("oracle_router_logits", "oracle_selected_softmax", "oracle_softmax_of_set",
                     "oracle_permute", "oracle_expert_combine", "oracle_moe_forward",
                     "oracle_route_scored", "oracle_moe_forward_scored"):
            getattr(lib, name).restype = i
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    return np.ascontiguousarray(a, dtype=dtype) if a is not None else None


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def router_logits(x, act_dtype: int, w_router, E: int, nthreads: int = 0) -> np.ndarray:
    x = _c(x)
    w_router = _c(w_router)
    T, d = x.shape
    out = np.empty((T, E), dtype=np.float64)
    _check(_load().oracle_router_logits(_p(x), act_dtype, T, d, _p(w_router), E, _p(out),
                                        nthreads), "router_logits")
    return out


def selected_softmax(logits, bias, k: int):
    logits = _c(logits, np.float64)
    T, E = logits.shape
    b = _c(bias, np.float32)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    _check(_load().oracle_selected_softmax(_p(logits), _p(b), T, E, k, _p(idx), _p(w),
                                           _p(margin)), "selected_softmax")
    return idx, w, margin


# scoring modes (oracle_route_scored): SelectedSoftmax, softmax before rank,
# sigmoid before rank
SELECTED_SOFTMAX, SOFTMAX, SIGMOID = 0, 1, 2


def route_scored(logits, bias, k: int, mode: int):
    """Routing in scoring mode `mode`: (topk_idx [T,k], topk_w [T,k], margin [T])."""
    logits = _c(logits, np.float64)
    T, E = logits.shape
    b = _c(bias, np.float32)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    _check(_load().oracle_route_scored(_p(logits), _p(b), T, E, k, mode, _p(idx), _p(w),
                                       _p(margin)), "route_scored")
    return idx, w, margin


def softmax_of_set(logits, topk_idx) -> np.ndarray:
    logits = _c(logits, np.float64)
    idx = _c(topk_idx, np.int32)
    T, E = logits.shape
    k = idx.shape[1]
    w = np.empty((T, k), dtype=np.float64)
    _check(_load().oracle_softmax_of_set(_p(logits), T, E, k, _p(idx), _p(w)), "softmax_of_set")
    return w


def permute(topk_idx, E: int):
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm_tok = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    _check(_load().oracle_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm_tok),
                                  _p(inv)), "permute")
    return counts, offsets, perm_tok, inv


def expert_combine(x, act_dtype: int, topk_idx, topk_w, w_gate, w_up, w_down, w_dtype: int,
                   E: int, F: int, nthreads: int = 0) -> np.ndarray:
    x = _c(x)
    T, d = x.shape
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float64)
    k = idx.shape[1]
    wg, wu, wd = _c(w_gate), _c(w_up), _c(w_down)
    out = np.empty((T, d), dtype=np.float64)
    _check(_load().oracle_expert_combine(_p(x), act_dtype, T, d, _p(idx), _p(w), k, _p(wg),
                                         _p(wu), _p(wd), w_dtype, E, F, _p(out), nthreads),
           "expert_combine")
    return out


def moe_forward(layer, nthreads: int = 0, mode: int = SELECTED_SOFTMAX):
    """Whole layer on a workloads.Layer in scoring mode `mode`.  Returns (out,
    topk_idx, topk_w, margin)."""
    x = _c(layer.x)
    T, d = x.shape
    E, k, F = layer.E, layer.k, layer.F
    out = np.empty((T, d), dtype=np.float64)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    wr, b = _c(layer.w_router), _c(layer.bias, np.float32)
    wg, wu, wd = _c(layer.w_gate), _c(layer.w_up), _c(layer.w_down)
    _check(_load().oracle_moe_forward_scored(_p(x), layer.act_dtype, T, d, _p(wr), _p(b), E, k,
                                             mode, _p(wg), _p(wu), _p(wd), layer.w_dtype, F,
                                             _p(out), _p(idx), _p(w), _p(margin), nthreads),
           "moe_forward")
    return out, idx, w, margin
