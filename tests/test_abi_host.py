"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/moe.h declares, and argument errors come back before any CUDA
call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from expert_routed_ffn_selectedsoftmax_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_bound_names():
    from expert_routed_ffn_selectedsoftmax_gb300 import binding
    assert declared_symbols() == sorted(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported(lib):
    """The .so exposes the moe_* ABI and nothing else that starts with moe_."""
    import subprocess
    from expert_routed_ffn_selectedsoftmax_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    names = {l.split()[-1] for l in out.stdout.splitlines() if l.strip()}
    moe = sorted(n for n in names if n.startswith("moe_"))
    assert moe == declared_symbols()


def test_status_strings_and_version(lib):
    for s in range(7):
        assert lib.moe_status_str(s)
    assert lib.moe_status_str(99) == b"unknown status"
    assert lib.moe_version() >= 100


def test_workspace_and_pack_sizes(lib):
    # invalid sizes -> 0
    assert lib.moe_workspace_size(8, 64, 8, 9, 128, 0, 0) == 0      # k > E
    assert lib.moe_workspace_size(8, 64, 8, 2, 128, 0, 2) == 0      # f32 act + q8 weights
    n = lib.moe_workspace_size(128, 1024, 64, 2, 512, 1, 1)
    # holds at least h (fp32 [T*k, F]) and the grouped bf16 rows [T*k, d]
    assert n >= 128 * 2 * 512 * 4 + 128 * 2 * 1024 * 2
    assert lib.moe_workspace_size(0, 64, 8, 2, 128, 0, 0) > 0
    assert lib.moe_q8_0_packed_size(10, 33) == 0
    assert lib.moe_q8_0_packed_size(3, 64) == 256 + 3 * 2 * 2


def test_argument_errors_are_synchronous(lib):
    vp = ctypes.c_void_p
    fake = vp(0x10000)         # never dereferenced: every call below fails validation first
    I, U = 1, 2                # MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED
    # k > E
    assert lib.moe_route(fake, 1, 4, 64, fake, None, 4, 5, fake, fake, None) == I
    # d not a multiple of 8
    assert lib.moe_route(fake, 1, 4, 60, fake, None, 4, 2, fake, fake, None) == I
    # unknown activation dtype
    assert lib.moe_route(fake, 7, 4, 64, fake, None, 4, 2, fake, fake, None) == I
    # E beyond the supported maximum
    assert lib.moe_route(fake, 1, 4, 64, fake, None, 300, 2, fake, fake, None) == U
    # misaligned x
    assert lib.moe_route(vp(0x10004), 1, 4, 64, fake, None, 4, 2, fake, fake, None) == I
    # permute: k > E, null outputs
    assert lib.moe_permute(fake, 4, 3, 2, fake, fake, fake, fake, None) == I
    assert lib.moe_permute(fake, 4, 1, 2, None, fake, fake, fake, None) == I
    assert lib.moe_permute(fake, 4, 1, 2, vp(0x10002), fake, fake, fake, None) == I   # misaligned
    # pack: cols not a multiple of 32, misaligned destination
    assert lib.moe_pack_q8_0(fake, 4, 48, fake, None) == I
    assert lib.moe_pack_q8_0(fake, 4, 64, vp(0x10010), None) == I
    args = dict(x=fake, act=1, T=4, d=256, wr=fake, b=None, E=8, k=2, wg=fake, wu=fake,
                wd=fake, wdt=1, F=128, out=fake, ws=fake, wsb=1 << 30, path=0)

    def fwd(**kw):
        a = dict(args, **kw)
        return lib.moe_forward(a["x"], a["act"], a["T"], a["d"], a["wr"], a["b"], a["E"], a["k"],
                               a["wg"], a["wu"], a["wd"], a["wdt"], a["F"], a["out"], a["ws"],
                               a["wsb"], a["path"], None)
    assert fwd(wsb=16) == 3                      # MOE_ERR_WORKSPACE
    assert fwd(F=100) == I                       # F % 8
    assert fwd(act=0, wdt=1) == U                # f32 activations with bf16 weights
    assert fwd(wdt=2, F=136) == I                # Q8_0 needs F % 32
    assert fwd(wdt=3, F=160) == I                # affine 4-bit needs F % 64
    assert fwd(wdt=3, d=192, path=2) == U        # affine 4-bit prefill GEMMs need d % 256
    assert fwd(act=0, wdt=3) == U                # affine 4-bit takes bf16 activations
    assert lib.moe_pack_q4_a64(fake, 4, 96, fake, None) == I      # cols % 64
    assert lib.moe_pack_q4_a64(fake, 4, 128, vp(0x10010), None) == I
    assert lib.moe_q4_a64_packed_size(4, 96) == 0
    # one row tile (rows padded to 128) x 2 groups, 4608 bytes per tile
    assert lib.moe_q4_a64_packed_size(4, 128) == 2 * 4608
    assert lib.moe_q4_a64_packed_size(129, 64) == 2 * 4608
    assert fwd(wdt=4, F=128) == I                # Q4_K needs whole 256-value super-blocks: F % 256
    assert fwd(wdt=4, d=384, F=256) == I         #   and d % 256
    assert fwd(act=0, wdt=4, F=256) == U         # Q4_K takes bf16 activations
    assert lib.moe_pack_q4_k(fake, 4, 192, fake, None) == I       # cols % 256
    assert lib.moe_pack_q4_k(fake, 4, 256, vp(0x10010), None) == I
    assert lib.moe_q4_k_packed_size(4, 192) == 0
    assert lib.moe_q4_k_packed_size(-1, 256) == 0
    # one row tile x 4 tile columns, 5120 bytes per tile (two scale/bias pairs a row)
    assert lib.moe_q4_k_packed_size(4, 256) == 4 * 5120
    assert lib.moe_q4_k_packed_size(129, 512) == 2 * 8 * 5120
    assert fwd(wdt=5, F=128) == I                # Q6_K: whole 256-value super-blocks
    assert fwd(act=0, wdt=5, F=256) == U         # Q6_K takes bf16 activations
    assert lib.moe_pack_q6_k(fake, 4, 192, fake, None) == I
    assert lib.moe_pack_q6_k(fake, 4, 256, vp(0x10010), None) == I
    assert lib.moe_q6_k_packed_size(4, 192) == 0
    # int8 plane (padded to 256 bytes), then fp16 scales, one per 16 values
    assert lib.moe_q6_k_packed_size(3, 256) == 768 + 3 * 16 * 2
    assert lib.moe_q6_k_packed_size(2, 512) == 1024 + 2 * 32 * 2
    assert fwd(act=0, wdt=6) == U                # fp8 takes bf16 activations
    assert fwd(wdt=6, wg=vp(0x10010)) == I       # fp8 packed buffers are 256-byte aligned
    assert fwd(wdt=7) == I                       # unknown weight storage
    assert lib.moe_pack_fp8(fake, 4, 0, fake, None) == I
    assert lib.moe_pack_fp8(fake, 4, 64, vp(0x10010), None) == I
    assert lib.moe_pack_fp8(fake, 0, 64, fake, None) == 0   # no rows: nothing to do
    assert lib.moe_fp8_packed_size(3, 0) == 0
    assert lib.moe_fp8_packed_size(-1, 64) == 0
    # E4M3 plane (padded to 256 bytes), then one fp32 scale per row
    assert lib.moe_fp8_packed_size(3, 64) == 256 + 3 * 4
    assert lib.moe_fp8_packed_size(130, 128) == 16640 + 130 * 4
    assert fwd(path=9) == I
    assert fwd(wg=None) == I
    assert fwd(ws=vp(0x10010)) == I              # workspace not 256-byte aligned
    assert fwd(act=0, wdt=0, path=2) == U        # prefill path needs bf16
    assert fwd(d=264, path=2) == U               # prefill path needs d % 256
    # T == 0 is a successful no-op that touches nothing
    assert fwd(T=0, wg=None, out=None, ws=None) == 0
    assert lib.moe_route(None, 1, 0, 64, None, None, 4, 2, None, None, None) == 0


def test_scoring_mode_is_checked_before_any_cuda_call(lib):
    """moe_route_scored / moe_forward_scored reject an unknown scoring mode
    (MOE_ERR_INVALID_ARG = 1) and accept the three defined ones on an empty
    batch (T = 0 returns before any launch)."""
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    for bad in (-1, 3, 99):
        assert lib.moe_route_scored(fake, 1, 4, 64, fake, None, 4, 2, bad, fake, fake, None) == 1
        assert lib.moe_forward_scored(fake, 1, 4, 64, fake, None, 4, 2, fake, fake, fake, 1, 128,
                                      fake, fake, 1 << 20, 0, bad, None, None) == 1
    for mode in (0, 1, 2):
        assert lib.moe_route_scored(None, 1, 0, 64, None, None, 4, 2, mode, None, None, None) == 0
        assert lib.moe_forward_scored(None, 1, 0, 64, None, None, 4, 2, None, None, None, 1, 128,
                                      None, None, 0, 0, mode, None, None) == 0


def test_ffn_dense_argument_checks(lib):
    """moe_ffn_dense: empty batch is a no-op; bad path / F / dtype rejected
    (MOE_ERR_INVALID_ARG = 1, MOE_ERR_UNSUPPORTED = 2) before any CUDA call."""
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    assert lib.moe_ffn_dense(None, 1, 0, 64, None, None, None, 1, 128, None, None, 0, 0, None) == 0
    assert lib.moe_ffn_dense(fake, 1, 4, 64, fake, fake, fake, 1, 128, fake, fake, 1 << 20, 9,
                             None) == 1
    assert lib.moe_ffn_dense(fake, 1, 4, 64, fake, fake, fake, 1, 100, fake, fake, 1 << 20, 0,
                             None) == 1
    assert lib.moe_ffn_dense(fake, 0, 4, 64, fake, fake, fake, 1, 128, fake, fake, 1 << 20, 0,
                             None) == 2


def test_debug_build_exports_the_debug_header_too():
    """libmoe_gb300_debug.so (MOE_DEBUG=1) exports the moe.h ABI plus the
    entry points of include/moe_debug.h; the release library does not export
    the latter."""
    import subprocess
    from expert_routed_ffn_selectedsoftmax_gb300 import build, binding
    dbg_header = os.path.join(ROOT, "include", "moe_debug.h")
    debug_names = sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", open(dbg_header).read())))
    assert debug_names == ["moe_debug_corrupt_next_offsets"]

    def exported(path):
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
        return sorted({ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[-1].startswith("moe_")})

    assert exported(build.build(debug=True)) == sorted(declared_symbols() + debug_names)
    assert exported(build.build()) == declared_symbols()

