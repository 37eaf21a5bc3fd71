"""Thin Python binding of the C ABI in include/moe.h (libmoe_gb300.so).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
the current stream); the functions carry the C names.  If the library has not
been built the first call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import build as _build

MOE_F32, MOE_BF16, MOE_Q8_0, MOE_Q4_A64, MOE_Q4_K, MOE_Q6_K, MOE_FP8 = 0, 1, 2, 3, 4, 5, 6
PACKED = (MOE_Q8_0, MOE_Q4_A64, MOE_Q4_K, MOE_Q6_K, MOE_FP8)   # storage types moe_forward takes repacked
MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL, MOE_PATH_DECODE_SIMT = 0, 1, 2, 3
MOE_SCORE_SELECTED_SOFTMAX, MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
          6: "MOE_ERR_DEVICE_CHECK"}

# Every symbol include/moe.h declares.
EXPORTS = ("moe_status_str", "moe_version", "moe_route", "moe_route_scored", "moe_permute",
           "moe_q8_0_packed_size", "moe_pack_q8_0", "moe_q4_a64_packed_size", "moe_pack_q4_a64",
           "moe_q4_k_packed_size", "moe_pack_q4_k", "moe_q6_k_packed_size", "moe_pack_q6_k",
           "moe_fp8_packed_size", "moe_pack_fp8",
           "moe_workspace_size", "moe_forward",
           "moe_forward_profiled", "moe_forward_scored", "moe_ffn_dense", "moe_forward_noalloc",
           "moe_workspace_views", "moe_forward_expire_wait", "moe_check", "moe_check_noalloc")

_lib = None
_debug_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({_lib.moe_status_str(status).decode() if _lib else ''})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libmoe_gb300.so and declare its signatures (raises if missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m expert_routed_ffn_selectedsoftmax_gb300.build)")
    _lib = _declare(ctypes.CDLL(path))
    return _lib


def load_debug_library():
    """The debug build (libmoe_gb300_debug.so, MOE_DEBUG=1: device-side checks
    of the grouping the expert kernels are given; include/moe_debug.h),
    compiled first if it is missing or stale.  A separate ctypes handle with
    the same signatures plus moe_debug_corrupt_next_offsets; the functions of
    this module keep using the release library."""
    global _debug_lib
    if _debug_lib is None:
        L = _declare(ctypes.CDLL(_build.build(debug=True)))
        L.moe_debug_corrupt_next_offsets.argtypes = []
        L.moe_debug_corrupt_next_offsets.restype = ctypes.c_int
        _debug_lib = L
    return _debug_lib


def _declare(L):
    vp, i, sz, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
    L.moe_status_str.argtypes = [i]
    L.moe_status_str.restype = ctypes.c_char_p
    L.moe_version.argtypes = []
    L.moe_version.restype = i
    L.moe_route.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp]
    L.moe_route.restype = i
    L.moe_route_scored.argtypes = [vp, i, i, i, vp, vp, i, i, i, vp, vp, vp]
    L.moe_route_scored.restype = i
    L.moe_permute.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp]
    L.moe_permute.restype = i
    L.moe_q8_0_packed_size.argtypes = [ll, i]
    L.moe_q8_0_packed_size.restype = sz
    L.moe_pack_q8_0.argtypes = [vp, ll, i, vp, vp]
    L.moe_pack_q8_0.restype = i
    L.moe_q4_a64_packed_size.argtypes = [ll, i]
    L.moe_q4_a64_packed_size.restype = sz
    L.moe_pack_q4_a64.argtypes = [vp, ll, i, vp, vp]
    L.moe_pack_q4_a64.restype = i
    L.moe_q4_k_packed_size.argtypes = [ll, i]
    L.moe_q4_k_packed_size.restype = sz
    L.moe_pack_q4_k.argtypes = [vp, ll, i, vp, vp]
    L.moe_pack_q4_k.restype = i
    L.moe_q6_k_packed_size.argtypes = [ll, i]
    L.moe_q6_k_packed_size.restype = sz
    L.moe_pack_q6_k.argtypes = [vp, ll, i, vp, vp]
    L.moe_pack_q6_k.restype = i
    L.moe_fp8_packed_size.argtypes = [ll, i]
    L.moe_fp8_packed_size.restype = sz
    L.moe_pack_fp8.argtypes = [vp, ll, i, vp, vp]
    L.moe_pack_fp8.restype = i
    L.moe_workspace_size.argtypes = [i, i, i, i, i, i, i]
    L.moe_workspace_size.restype = sz
    L.moe_forward.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, vp, vp, sz, i, vp]
    L.moe_forward.restype = i
    L.moe_forward_profiled.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, vp, vp, sz,
                                       i, vp, vp]
    L.moe_forward_profiled.restype = i
    L.moe_forward_scored.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, vp, vp, sz,
                                     i, i, vp, vp]
    L.moe_forward_scored.restype = i
    L.moe_ffn_dense.argtypes = [vp, i, i, i, vp, vp, vp, i, i, vp, vp, sz, i, vp]
    L.moe_ffn_dense.restype = i
    L.moe_forward_noalloc.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, vp, i, vp]
    L.moe_forward_noalloc.restype = i
    L.moe_forward_expire_wait.argtypes = [vp, i, i, i, vp, vp, i, i, vp, vp, vp, i, i, vp, vp, sz,
                                          i, i, ctypes.c_uint32, vp]
    L.moe_forward_expire_wait.restype = i
    L.moe_workspace_views.argtypes = [i, i, i, i, i, i, i, vp]
    L.moe_workspace_views.restype = i
    L.moe_check.argtypes = [vp, vp, vp]
    L.moe_check.restype = i
    L.moe_check_noalloc.argtypes = [vp, vp]
    L.moe_check_noalloc.restype = i
    return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _act_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def moe_route(x: torch.Tensor, w_router: torch.Tensor, sel_bias: Optional[torch.Tensor], k: int,
              topk_idx: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
              scoring: int = MOE_SCORE_SELECTED_SOFTMAX):
    """Router projection + scoring (SelectedSoftmax by default) -> (topk_idx int32
    [T,k], topk_w fp32 [T,k])."""
    L = load_library()
    T, d = x.shape
    E = w_router.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    if scoring == MOE_SCORE_SELECTED_SOFTMAX:
        _check(L.moe_route(_ptr(x), _act_dtype(x), T, d, _ptr(w_router), _ptr(sel_bias), E, k,
                           _ptr(topk_idx), _ptr(topk_w), _stream(x)), "moe_route")
    else:
        _check(L.moe_route_scored(_ptr(x), _act_dtype(x), T, d, _ptr(w_router), _ptr(sel_bias),
                                  E, k, scoring, _ptr(topk_idx), _ptr(topk_w), _stream(x)),
               "moe_route_scored")
    return topk_idx, topk_w


def moe_permute(topk_idx: torch.Tensor, E: int):
    """Token grouping -> (counts [E], offsets [E+1], perm_tok [T*k], inv [T*k]), int32."""
    L = load_library()
    T, k = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm_tok = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    _check(L.moe_permute(_ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm_tok),
                         _ptr(inv), _stream(topk_idx)), "moe_permute")
    return counts, offsets, perm_tok[:T * k], inv[:T * k]


def moe_q8_0_packed_size(rows: int, cols: int) -> int:
    return int(load_library().moe_q8_0_packed_size(rows, cols))


def moe_pack_q8_0(blocks: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Repack Q8_0 blocks (uint8 device tensor, rows*cols/32*34 bytes) into planes."""
    L = load_library()
    n = moe_q8_0_packed_size(rows, cols)
    if n == 0 and rows != 0:
        raise MoeError(1, "moe_q8_0_packed_size")
    packed = torch.empty(max(n, 256), dtype=torch.uint8, device=blocks.device)
    _check(L.moe_pack_q8_0(_ptr(blocks), rows, cols, _ptr(packed), _stream(blocks)),
           "moe_pack_q8_0")
    return packed


def moe_q4_a64_packed_size(rows: int, cols: int) -> int:
    return int(load_library().moe_q4_a64_packed_size(rows, cols))


def moe_pack_q4_a64(blocks: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Repack affine 4-bit group-64 blocks (uint8 device tensor, rows*cols/64*36
    bytes) into the tiles moe_forward takes."""
    L = load_library()
    n = moe_q4_a64_packed_size(rows, cols)
    if n == 0 and rows != 0:
        raise MoeError(1, "moe_q4_a64_packed_size")
    packed = torch.empty(max(n, 256), dtype=torch.uint8, device=blocks.device)
    _check(L.moe_pack_q4_a64(_ptr(blocks), rows, cols, _ptr(packed), _stream(blocks)),
           "moe_pack_q4_a64")
    return packed


def moe_q4_k_packed_size(rows: int, cols: int) -> int:
    return int(load_library().moe_q4_k_packed_size(rows, cols))


def moe_pack_q4_k(blocks: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Repack Q4_K super-blocks (uint8 device tensor, rows*cols/256*144 bytes)
    into the tiles moe_forward takes."""
    L = load_library()
    n = moe_q4_k_packed_size(rows, cols)
    if n == 0 and rows != 0:
        raise MoeError(1, "moe_q4_k_packed_size")
    packed = torch.empty(max(n, 256), dtype=torch.uint8, device=blocks.device)
    _check(L.moe_pack_q4_k(_ptr(blocks), rows, cols, _ptr(packed), _stream(blocks)),
           "moe_pack_q4_k")
    return packed


def moe_q6_k_packed_size(rows: int, cols: int) -> int:
    return int(load_library().moe_q6_k_packed_size(rows, cols))


def moe_pack_q6_k(blocks: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Repack Q6_K super-blocks (uint8 device tensor, rows*cols/256*210 bytes)
    into the 8-bit planes moe_forward takes."""
    L = load_library()
    n = moe_q6_k_packed_size(rows, cols)
    if n == 0 and rows != 0:
        raise MoeError(1, "moe_q6_k_packed_size")
    packed = torch.empty(max(n, 256), dtype=torch.uint8, device=blocks.device)
    _check(L.moe_pack_q6_k(_ptr(blocks), rows, cols, _ptr(packed), _stream(blocks)),
           "moe_pack_q6_k")
    return packed


def moe_fp8_packed_size(rows: int, cols: int) -> int:
    return int(load_library().moe_fp8_packed_size(rows, cols))


def moe_pack_fp8(rows_in: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Repack fp8 rows {fp32 scale, E4M3 codes} (uint8 device tensor,
    rows*(4+cols) bytes) into the E4M3 plane and row scales moe_forward takes."""
    L = load_library()
    n = moe_fp8_packed_size(rows, cols)
    if n == 0 and rows != 0:
        raise MoeError(1, "moe_fp8_packed_size")
    packed = torch.empty(max(n, 256), dtype=torch.uint8, device=rows_in.device)
    _check(L.moe_pack_fp8(_ptr(rows_in), rows, cols, _ptr(packed), _stream(rows_in)),
           "moe_pack_fp8")
    return packed


def moe_workspace_size(T: int, d: int, E: int, k: int, F: int, act_dt: int, w_dt: int) -> int:
    return int(load_library().moe_workspace_size(T, d, E, k, F, act_dt, w_dt))


def moe_forward(x: torch.Tensor, w_router: torch.Tensor, sel_bias: Optional[torch.Tensor],
                w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor, k: int,
                F: Optional[int] = None, w_dtype: Optional[int] = None,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                path: int = MOE_PATH_AUTO, events=None,
                scoring: int = MOE_SCORE_SELECTED_SOFTMAX) -> torch.Tensor:
    """The whole MoE layer -> out fp32 [T, d].

    Weights: float32/bfloat16 tensors [E,F,d], [E,F,d], [E,d,F]; or, with
    w_dtype=MOE_Q8_0 / MOE_Q4_A64 / MOE_Q4_K / MOE_Q6_K / MOE_FP8, uint8 buffers from
    moe_pack_q8_0 / moe_pack_q4_a64 / moe_pack_q4_k / moe_pack_q6_k / moe_pack_fp8 (then F is
    required).
    events: optional sequence of 6 torch.cuda.Event(enable_timing=True), recorded
    at the stage boundaries (moe_forward_profiled).
    scoring: a MOE_SCORE_* mode (moe_forward_scored when not SelectedSoftmax).
    """
    L = load_library()
    T, d = x.shape
    E = w_router.shape[0]
    act = _act_dtype(x)
    if w_dtype is None:
        w_dtype = _act_dtype(w_gate)
    if F is None:
        if w_dtype in PACKED:
            raise ValueError("F is required for block-quantised weights")
        F = w_gate.shape[1]
    if out is None:
        out = torch.empty((T, d), dtype=torch.float32, device=x.device)
    ws_bytes = moe_workspace_size(T, d, E, k, F, act, w_dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    ws_len = workspace.numel() * workspace.element_size()
    if scoring != MOE_SCORE_SELECTED_SOFTMAX:
        handles = None
        if events is not None:
            if len(events) != 6:
                raise ValueError("events: 6 CUDA events expected")
            handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
        _check(L.moe_forward_scored(_ptr(x), act, T, d, _ptr(w_router), _ptr(sel_bias), E, k,
                                    _ptr(w_gate), _ptr(w_up), _ptr(w_down), w_dtype, F,
                                    _ptr(out), _ptr(workspace), ws_len, path, scoring, handles,
                                    _stream(x)), "moe_forward_scored")
    elif events is None:
        _check(L.moe_forward(_ptr(x), act, T, d, _ptr(w_router), _ptr(sel_bias), E, k,
                             _ptr(w_gate), _ptr(w_up), _ptr(w_down), w_dtype, F, _ptr(out),
                             _ptr(workspace), ws_len, path, _stream(x)), "moe_forward")
    else:
        if len(events) != 6:
            raise ValueError("events: 6 CUDA events expected")
        handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
        _check(L.moe_forward_profiled(_ptr(x), act, T, d, _ptr(w_router), _ptr(sel_bias), E, k,
                                      _ptr(w_gate), _ptr(w_up), _ptr(w_down), w_dtype, F,
                                      _ptr(out), _ptr(workspace), ws_len, path, handles,
                                      _stream(x)), "moe_forward_profiled")
    return out


def moe_ffn_dense(x: torch.Tensor, w_gate: torch.Tensor, w_up: torch.Tensor,
                  w_down: torch.Tensor, F: Optional[int] = None, w_dtype: Optional[int] = None,
                  out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  path: int = MOE_PATH_AUTO) -> torch.Tensor:
    """A dense SwiGLU FFN layer -> out fp32 [T, d].

    Weights: float32/bfloat16 tensors [F,d], [F,d], [d,F] (or [1,F,d] ...); or,
    with w_dtype=MOE_Q8_0 / MOE_Q4_A64 / MOE_Q4_K / MOE_Q6_K / MOE_FP8, uint8 buffers from
    moe_pack_q8_0 / moe_pack_q4_a64 / moe_pack_q4_k / moe_pack_q6_k / moe_pack_fp8 (then F is
    required).
    """
    L = load_library()
    T, d = x.shape
    act = _act_dtype(x)
    if w_dtype is None:
        w_dtype = _act_dtype(w_gate)
    if F is None:
        if w_dtype in PACKED:
            raise ValueError("F is required for block-quantised weights")
        F = w_gate.shape[-2]
    if out is None:
        out = torch.empty((T, d), dtype=torch.float32, device=x.device)
    ws_bytes = moe_workspace_size(T, d, 1, 1, F, act, w_dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    ws_len = workspace.numel() * workspace.element_size()
    _check(L.moe_ffn_dense(_ptr(x), act, T, d, _ptr(w_gate), _ptr(w_up), _ptr(w_down), w_dtype, F,
                           _ptr(out), _ptr(workspace), ws_len, path, _stream(x)), "moe_ffn_dense")
    return out


def moe_forward_noalloc(x: torch.Tensor, w_router: torch.Tensor,
                        sel_bias: Optional[torch.Tensor], w_gate: torch.Tensor,
                        w_up: torch.Tensor, w_down: torch.Tensor, k: int, out: torch.Tensor,
                        F: Optional[int] = None, w_dtype: Optional[int] = None,
                        path: int = MOE_PATH_AUTO) -> torch.Tensor:
    """moe_forward without a workspace: the library's static scratch is used.

    For hosts that cannot allocate device memory; `out` must be supplied.
    Layers needing more than 8 MiB of scratch raise MOE_ERR_WORKSPACE.
    """
    L = load_library()
    T, d = x.shape
    E = w_router.shape[0]
    if w_dtype is None:
        w_dtype = _act_dtype(w_gate)
    if F is None:
        if w_dtype in PACKED:
            raise ValueError("F is required for block-quantised weights")
        F = w_gate.shape[1]
    _check(L.moe_forward_noalloc(_ptr(x), _act_dtype(x), T, d, _ptr(w_router), _ptr(sel_bias), E,
                                 k, _ptr(w_gate), _ptr(w_up), _ptr(w_down), w_dtype, F, _ptr(out),
                                 path, _stream(x)), "moe_forward_noalloc")
    return out


VIEW_NAMES = ("topk_idx", "topk_w", "counts", "offsets", "perm_tok", "inv", "perm_w")


def moe_workspace_views(T: int, d: int, E: int, k: int, F: int, act_dt: int, w_dt: int) -> dict:
    """Byte offsets of the routing / grouping arrays a layer call leaves in its
    workspace: {name: offset} for VIEW_NAMES."""
    L = load_library()
    views = (ctypes.c_size_t * 7)()
    _check(L.moe_workspace_views(T, d, E, k, F, act_dt, w_dt, views), "moe_workspace_views")
    return dict(zip(VIEW_NAMES, [int(v) for v in views]))


def read_routing(workspace: torch.Tensor, T: int, d: int, E: int, k: int, F: int, act_dt: int,
                 w_dt: int) -> dict:
    """The routing and grouping a layer call wrote into `workspace` (read after
    the call's stream work completed): views of the workspace bytes, as
    torch tensors on its device."""
    off = moe_workspace_views(T, d, E, k, F, act_dt, w_dt)
    n = T * k
    shapes = {"topk_idx": ((T, k), torch.int32), "topk_w": ((T, k), torch.float32),
              "counts": ((E,), torch.int32), "offsets": ((E + 1,), torch.int32),
              "perm_tok": ((n,), torch.int32), "inv": ((n,), torch.int32),
              "perm_w": ((n,), torch.float32)}
    out = {}
    for name, (shape, dt) in shapes.items():
        count = int(np.prod(shape))
        raw = workspace[off[name]:off[name] + 4 * count]
        out[name] = raw.view(dt).reshape(shape)
    return out


def moe_check_noalloc() -> int:
    """moe_check for moe_forward_noalloc's static scratch on the current device."""
    L = load_library()
    word = ctypes.c_uint32(0)
    _check(L.moe_check_noalloc(ctypes.byref(word), _stream_current()), "moe_check_noalloc")
    return word.value


def _stream_current():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def moe_check(workspace: torch.Tensor) -> int:
    """Wait for the current stream, return the device status word (raises on error)."""
    L = load_library()
    word = ctypes.c_uint32(0)
    _check(L.moe_check(_ptr(workspace), ctypes.byref(word), _stream(workspace)), "moe_check")
    return word.value
