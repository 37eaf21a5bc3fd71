"""Failure handling on the GPU without a fault: bounded waits that give up.

Every wait of the library's tensor-core kernels is bounded.  The test hook
moe_forward_expire_wait makes one wait of one kernel family -- on a barrier
that nothing ever arrives on and that no copy or MMA targets -- give up after
a short limit, in every CTA of that kernel.  The kernel must then return (no
hang: moe_check synchronises), report MOE_ERR_TIMEOUT through the status word,
and leave the device usable: a normal call right after on the same workspace
is clean and matches the oracle.  Nothing here faults, traps or waits without
a bound.
"""
import ctypes
import time

import numpy as np
import pytest

import oracle
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

from helpers import check_output, gpu_forward_views, upload_layer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DECODE, PREFILL = 1, 2
ROUTER_CLUSTER, ROUTER_TC, DECODE_SPLIT, DECODE_FUSED, GEMM = 1, 2, 3, 4, 5
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_TIMEOUT = 0, 1, 2, 5
WAIT_NS = 1_000_000   # 1 ms


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg.load_library()


def _expire(lib, layer, t, ws, out, path, family, wait_ns=WAIT_NS):
    p = lambda a: ctypes.c_void_p(a.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_forward_expire_wait(
        p(t["x"]), layer.act_dtype, layer.T, layer.d, p(t["w_router"]), p(t["bias"]), layer.E,
        layer.k, p(t["w_gate"]), p(t["w_up"]), p(t["w_down"]), layer.w_dtype, layer.F, p(out),
        p(ws), ws.numel(), path, family, ctypes.c_uint32(wait_ns), stream)


CASES = [
    # (family, path, (T, d, E, k, F), weights)
    (ROUTER_CLUSTER, DECODE, (32, 256, 8, 2, 128), wl.BF16),
    (ROUTER_TC, PREFILL, (600, 256, 8, 2, 128), wl.BF16),
    (DECODE_SPLIT, DECODE, (32, 256, 8, 2, 128), wl.BF16),
    (DECODE_SPLIT, DECODE, (32, 256, 8, 4, 128), wl.BF16),     # k > 2
    (DECODE_SPLIT, DECODE, (8, 256, 8, 1, 128), wl.Q4_A64),    # 4-bit converter warps
    (DECODE_SPLIT, DECODE, (8, 256, 8, 1, 256), wl.Q8_0),      # 8-bit converter warps
    (DECODE_SPLIT, DECODE, (8, 256, 8, 1, 256), wl.FP8),       # fp8 converter warps
    (DECODE_FUSED, DECODE, (128, 256, 64, 2, 512), wl.BF16),
    (GEMM, PREFILL, (600, 256, 4, 2, 128), wl.BF16),
    (GEMM, PREFILL, (600, 256, 4, 2, 128), wl.Q8_0),   # CTA pairs (clusters of two)
    (GEMM, PREFILL, (600, 256, 4, 2, 128), wl.FP8),
]


@pytest.mark.parametrize("family,path,shape,wdt", CASES)
def test_expired_wait_reports_timeout_and_the_next_call_is_clean(lib, family, path, shape, wdt):
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    T, d, E, k, F = shape
    layer = wl.make_custom_layer(41, T=T, d=d, E=E, k=k, F=F, act_dtype=wl.BF16, w_dtype=wdt,
                                 bias_sd=0.5)
    t = upload_layer(layer, DEV)
    ws = torch.empty(pkg.moe_workspace_size(T, d, E, k, F, 1, wdt), dtype=torch.uint8, device=DEV)
    out = torch.empty((T, d), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _expire(lib, layer, t, ws, out, path, family) == MOE_OK
    word = ctypes.c_uint32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.moe_check(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(word), stream)
    elapsed = time.perf_counter() - t0
    assert st == MOE_ERR_TIMEOUT, f"moe_check {st}, word {word.value}"
    assert word.value & 1
    assert elapsed < 10.0          # returned (bounded), well inside the 2 s limit per wait
    # the context is usable and the same workspace gives a clean, correct call
    o2, r = gpu_forward_views(layer, DEV, path=path, t=t)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(o2, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])
    gpu_forward = pkg.moe_forward(t["x"], t["w_router"], t["bias"], t["w_gate"], t["w_up"],
                                  t["w_down"], k, F=F, w_dtype=wdt, path=path, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.moe_check(ws) == 0
    assert np.array_equal(gpu_forward.cpu().numpy(), o2)


def test_hook_arguments(lib):
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(42, T=32, d=256, E=8, k=2, F=128, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    t = upload_layer(layer, DEV)
    ws = torch.empty(pkg.moe_workspace_size(32, 256, 8, 2, 128, 1, 1), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty((32, 256), dtype=torch.float32, device=DEV)
    assert _expire(lib, layer, t, ws, out, DECODE, 0) == MOE_ERR_INVALID_ARG
    assert _expire(lib, layer, t, ws, out, DECODE, 6) == MOE_ERR_INVALID_ARG
    assert _expire(lib, layer, t, ws, out, DECODE, ROUTER_CLUSTER, 0) == MOE_ERR_INVALID_ARG
    # a family that does not run for these arguments: nothing is enqueued
    assert _expire(lib, layer, t, ws, out, DECODE, GEMM) == MOE_ERR_UNSUPPORTED
    assert _expire(lib, layer, t, ws, out, DECODE, ROUTER_TC) == MOE_ERR_UNSUPPORTED
