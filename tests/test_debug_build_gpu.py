"""The debug build (libmoe_gb300_debug.so, MOE_DEBUG=1; include/moe_debug.h):
its device-side checks of the grouping the expert kernels are given change no
result, and an inconsistent grouping is reported, not used.

The inconsistency is made on purpose but safely: moe_debug_corrupt_next_offsets
makes the next call add 1 to offsets[E] in its own workspace after grouping (a
store inside the workspace); every expert kernel then finds offsets that do not
end at T*k, does no work and records MOE_ERR_DEVICE_CHECK.  No kernel reads or
writes out of bounds on that path, and the next call on the same workspace is
clean."""
import ctypes

import numpy as np
import pytest

from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

from helpers import upload_layer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DECODE, PREFILL, SIMT = 1, 2, 3
DEVICE_CHECK = 6   # MOE_ERR_DEVICE_CHECK

# (act, w, T, d, E, k, F, path): the one-launch decode kernel, the split-K
# tensor-core decode kernels (bf16, 4-bit and fp8, k = 4 through the combine), the
# CUDA-core kernels, and the grouped GEMMs (bf16, Q8_0, 4-bit, fp8)
CASES = [
    (wl.BF16, wl.BF16, 128, 1024, 64, 2, 512, 0),
    (wl.BF16, wl.BF16, 40, 512, 16, 2, 384, DECODE),
    (wl.BF16, wl.Q4_A64, 64, 512, 16, 1, 384, DECODE),
    (wl.BF16, wl.BF16, 64, 512, 16, 4, 384, DECODE),
    (wl.F32, wl.F32, 37, 256, 8, 2, 128, SIMT),
    (wl.BF16, wl.Q8_0, 20, 256, 8, 2, 256, SIMT),
    (wl.BF16, wl.BF16, 600, 256, 8, 2, 256, PREFILL),
    (wl.BF16, wl.Q8_0, 600, 256, 8, 2, 256, PREFILL),
    (wl.BF16, wl.Q4_A64, 600, 256, 8, 2, 256, PREFILL),
    (wl.BF16, wl.FP8, 64, 512, 16, 1, 384, DECODE),
    (wl.BF16, wl.FP8, 600, 256, 8, 2, 256, PREFILL),
]


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg.load_library(), pkg.binding.load_debug_library()


def _forward(L, layer, t, out, ws, path):
    p = lambda a: ctypes.c_void_p(a.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.moe_forward(p(t["x"]), layer.act_dtype, layer.T, layer.d, p(t["w_router"]), p(t["bias"]),
                         layer.E, layer.k, p(t["w_gate"]), p(t["w_up"]), p(t["w_down"]),
                         layer.w_dtype, layer.F, p(out), p(ws), ws.numel(), path, stream)


def _check(L, ws):
    w = ctypes.c_uint32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.moe_check(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(w), stream)


def _setup(rel, case, seed):
    act, wdt, T, d, E, k, F, path = case
    layer = wl.make_custom_layer(seed, T=T, d=d, E=E, k=k, F=F, act_dtype=act, w_dtype=wdt, bias_sd=0.5)
    t = upload_layer(layer, DEV)
    ws = torch.empty(rel.moe_workspace_size(T, d, E, k, F, act, wdt), dtype=torch.uint8, device=DEV)
    return layer, t, ws, path


@pytest.mark.parametrize("case", CASES)
def test_debug_build_gives_the_release_results(libs, case):
    rel, dbg = libs
    layer, t, ws, path = _setup(rel, case, 41)
    outs = []
    for L in (rel, dbg):
        out = torch.full((layer.T, layer.d), float("nan"), dtype=torch.float32, device=DEV)
        assert _forward(L, layer, t, out, ws, path) == 0
        torch.cuda.synchronize()
        assert _check(L, ws) == 0
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("case", CASES)
def test_debug_build_reports_inconsistent_offsets(libs, case):
    rel, dbg = libs
    layer, t, ws, path = _setup(rel, case, 42)
    out = torch.zeros((layer.T, layer.d), dtype=torch.float32, device=DEV)
    assert dbg.moe_debug_corrupt_next_offsets() == 0
    assert _forward(dbg, layer, t, out, ws, path) == 0   # launches; the checks report on the device
    torch.cuda.synchronize()
    assert _check(dbg, ws) == DEVICE_CHECK
    # the next call on the same workspace is clean and equals the release build's
    a = torch.full_like(out, float("nan"))
    b = torch.full_like(out, float("nan"))
    assert _forward(dbg, layer, t, a, ws, path) == 0
    torch.cuda.synchronize()
    assert _check(dbg, ws) == 0
    assert _forward(rel, layer, t, b, ws, path) == 0
    torch.cuda.synchronize()
    assert torch.equal(a, b)
