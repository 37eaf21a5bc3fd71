"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars: routing indices and token grouping bit-exact (indices wherever the
oracle's ranking margin is >= 1e-3); routing weights within 2e-6; outputs with
max|err| <= 1e-4 * RMS(ref) for fp32 and <= 2e-2 * RMS(ref) for bf16 / Q8_0.
"""
import numpy as np
import pytest

import oracle
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

from helpers import (MARGIN, check_output, check_routing_views, compare_routing, gpu_forward,
                     gpu_forward_views, to_dev, upload_layer)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DECODE, PREFILL, SIMT = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    pkg.load_library()
    torch.cuda.set_device(0)


def _route(layer):
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    x, wr, b = to_dev(layer.x, DEV), to_dev(layer.w_router, DEV), to_dev(layer.bias, DEV)
    idx, w = pkg.moe_route(x, wr, b, layer.k)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def _oracle_route(layer):
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    return oracle.selected_softmax(logits, layer.bias, layer.k)


# ------------------------------------------------------------------ routing
ROUTE_CASES = [
    ("tiny_fp32", None), ("zonos3_mini_decode", None), ("zonos2_decode", 1),
    ("zonos2_decode", 8), ("zonos2_decode", 64), ("zonos3_mini_prefill", None),
    ("zonos2_prefill_q8", None),
]


@pytest.mark.parametrize("seed", [1, 7, 13])
@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_route_matches_oracle(name, T, seed):
    w = wl.WORKLOADS[name]
    # only x, W_r and the bias matter for routing: draw a small-F layer
    layer = wl.make_layer(w, seed=seed, T=T, F=32)
    idx, wts = _route(layer)
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    idx_ref, w_ref, margin = oracle.selected_softmax(logits, layer.bias, layer.k)
    ok = compare_routing(idx, wts, idx_ref, w_ref, margin, layer.k, logits=logits,
                         bias=layer.bias)
    assert ok.mean() > 0.95


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 3, 3), (33, 2, 64), (300, 4, 256), (1000, 8, 16)])
def test_route_edge_shapes(T, k, E):
    layer = wl.make_custom_layer(7, T=T, d=64, E=E, k=k, F=32, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16, bias_sd=0.3)
    idx, wts = _route(layer)
    idx_ref, w_ref, margin = _oracle_route(layer)
    compare_routing(idx, wts, idx_ref, w_ref, margin, k)
    assert np.all(np.abs(wts.sum(1) - 1) < 1e-6)


def test_route_ties_go_to_lower_index():
    """Experts 1, 2, 3 share one router row (equal logits); 0, 4, 5 its negation."""
    layer = wl.make_custom_layer(3, T=16, d=64, E=6, k=2, F=32, act_dtype=wl.F32,
                                 w_dtype=wl.F32, bias_sd=0.0)
    v = layer.w_router[0].copy()
    layer.w_router[[1, 2, 3]] = v
    layer.w_router[[0, 4, 5]] = -v
    layer.x = (np.outer(np.arange(1, 17), v) * 4).astype(np.float32)   # x . v > 0
    idx, wts = _route(layer)
    assert np.all(idx == [1, 2])
    assert np.all(wts == 0.5)


@pytest.mark.parametrize("T", [16, 200, 600])
def test_route_ties_go_to_lower_index_bf16(T):
    """Same on the bf16 (tensor-core) router: identical router rows give
    bitwise-equal logits, and the lower expert index wins."""
    layer = wl.make_custom_layer(4, T=T, d=128, E=6, k=2, F=32, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16, bias_sd=0.0)
    v = layer.w_router[0].copy()
    neg = wl.f32_to_bf16_bits(-wl.bf16_bits_to_f32(v))
    layer.w_router[[1, 2, 3]] = v
    layer.w_router[[0, 4, 5]] = neg
    xv = wl.bf16_bits_to_f32(v)
    layer.x = wl.f32_to_bf16_bits(np.outer(np.linspace(1, 2, T), xv) * 4)
    idx, wts = _route(layer)
    assert np.all(idx == [1, 2])
    assert np.all(wts == 0.5)


# ------------------------------------------------------------------ permute
@pytest.mark.parametrize("T,k,E", [(0, 2, 4), (1, 1, 1), (128, 2, 64), (8192, 2, 64),
                                   (4096, 1, 16), (777, 3, 250), (40000, 8, 256)])
def test_permute_bit_exact(T, k, E):
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rng = np.random.default_rng(T + k + E)
    if T:
        # skewed choice: distinct experts per token, biased toward low ids
        p = 1.0 / np.arange(1, E + 1)
        p /= p.sum()
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        idx = np.zeros((0, k), np.int32)
    counts, offsets, perm_tok, inv = pkg.moe_permute(to_dev(idx, DEV), E)
    torch.cuda.synchronize()
    c_ref, o_ref, p_ref, i_ref = oracle.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(offsets.cpu().numpy(), o_ref)
    assert np.array_equal(perm_tok.cpu().numpy(), p_ref)
    assert np.array_equal(inv.cpu().numpy(), i_ref)


# ------------------------------------------------- whole layer, small sizes
SMALL = [
    # (act, w, T, d, E, k, F)  -- several tiles and ragged tails
    (wl.F32, wl.F32, 8, 64, 8, 2, 128),
    (wl.F32, wl.F32, 37, 200, 7, 3, 72),
    (wl.BF16, wl.BF16, 1, 256, 8, 2, 128),
    (wl.BF16, wl.BF16, 61, 264, 12, 2, 136),
    (wl.BF16, wl.BF16, 200, 512, 16, 1, 384),
    (wl.BF16, wl.Q8_0, 45, 256, 8, 2, 160),
    (wl.BF16, wl.Q8_0, 3, 2048, 16, 1, 2816),
    (wl.BF16, wl.BF16, 96, 256, 4, 4, 128),     # k == E: dense gating
    (wl.BF16, wl.Q4_A64, 5, 256, 8, 2, 128),    # affine 4-bit experts (tensor-core decode:
    (wl.BF16, wl.Q4_A64, 70, 512, 16, 1, 192),  #   tiles converted in shared memory; F=192: CUDA cores)
    (wl.BF16, wl.Q4_A64, 33, 256, 16, 2, 256),
    (wl.BF16, wl.Q4_A64, 128, 1024, 64, 2, 512),
    (wl.BF16, wl.Q4_A64, 300, 512, 16, 4, 384),
    (wl.BF16, wl.Q4_K, 5, 256, 8, 2, 256),      # Q4_K experts: two (scale, bias) pairs per
    (wl.BF16, wl.Q4_K, 70, 512, 16, 1, 256),    #   tile row, whole 256-value super-blocks
    (wl.BF16, wl.Q4_K, 128, 1024, 64, 2, 512),
    (wl.BF16, wl.Q4_K, 300, 512, 16, 4, 768),
    (wl.BF16, wl.Q6_K, 5, 256, 8, 2, 256),      # Q6_K experts: 8-bit planes, a scale per 16
    (wl.BF16, wl.Q6_K, 70, 512, 16, 1, 512),    #   values (CUDA-core decode kernels)
    (wl.BF16, wl.Q6_K, 33, 1024, 64, 2, 256),
    (wl.BF16, wl.FP8, 5, 256, 8, 2, 128),       # fp8 experts: E4M3 planes, a scale per row
    (wl.BF16, wl.FP8, 70, 512, 16, 1, 192),     #   (F = 192: CUDA-core decode kernels)
    (wl.BF16, wl.FP8, 33, 1024, 64, 2, 256),
    (wl.BF16, wl.FP8, 300, 512, 16, 4, 384),
    (wl.BF16, wl.BF16, 5, 512, 64, 8, 128),     # few tokens: largest E and k of the small-batch router
    (wl.BF16, wl.BF16, 8, 2048, 33, 3, 128),    # few tokens: ragged E, longest rows
    (wl.BF16, wl.BF16, 40, 256, 256, 8, 128),   # the largest E and k the library takes
    (wl.F32, wl.F32, 20, 64, 256, 8, 64),
]


@pytest.mark.parametrize("path", [DECODE, SIMT])
@pytest.mark.parametrize("act,wdt,T,d,E,k,F", SMALL)
def test_forward_small_matches_oracle(act, wdt, T, d, E, k, F, path):
    layer = wl.make_custom_layer(11, T=T, d=d, E=E, k=k, F=F, act_dtype=act, w_dtype=wdt,
                                 bias_sd=0.3)
    out, r = gpu_forward_views(layer, DEV, path=path)
    check_routing_views(r, layer)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("path", [DECODE, SIMT])
def test_forward_all_tokens_one_expert(path):
    """A bias that sends every token to expert 3 (and 5): many row blocks in one expert."""
    layer = wl.make_custom_layer(12, T=150, d=256, E=8, k=2, F=128, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    layer.bias[:] = 0
    layer.bias[3] = 100.0
    layer.bias[5] = 50.0
    out = gpu_forward(layer, DEV, path=path)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    assert np.all(idx_ref == [3, 5])
    check_output(out.cpu().numpy(), layer, ref, idx_ref, margin)


def test_forward_empty_batch():
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(13, T=0, d=64, E=4, k=2, F=64, act_dtype=wl.F32,
                                 w_dtype=wl.F32)
    t = upload_layer(layer, DEV)
    out = pkg.moe_forward(t["x"], t["w_router"], t["bias"], t["w_gate"], t["w_up"], t["w_down"], 2)
    assert out.shape == (0, 64)


def test_forward_no_bias_pointer():
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(14, T=20, d=128, E=8, k=2, F=64, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    t = upload_layer(layer, DEV)
    out = pkg.moe_forward(t["x"], t["w_router"], None, t["w_gate"], t["w_up"], t["w_down"], 2)
    layer.bias[:] = 0
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(out.cpu().numpy(), layer, ref, idx_ref, margin)


# ------------------------------------------------------------- properties
def test_deterministic_and_permutation_equivariant():
    layer = wl.make_custom_layer(15, T=64, d=256, E=16, k=2, F=128, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    t = upload_layer(layer, DEV)
    a = gpu_forward(layer, DEV, t=t).cpu().numpy()
    b = gpu_forward(layer, DEV, t=t).cpu().numpy()
    assert np.array_equal(a, b)
    perm = np.random.default_rng(0).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])


def test_k1_weights_exactly_one_and_bias_only_selects():
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(16, T=100, d=128, E=8, k=3, F=64, act_dtype=wl.F32,
                                 w_dtype=wl.F32)
    x, wr = to_dev(layer.x, DEV), to_dev(layer.w_router, DEV)
    _, w1 = pkg.moe_route(x, wr, None, 1)
    assert torch.all(w1 == 1.0)
    idx0, w0 = pkg.moe_route(x, wr, None, 3)
    # bias forcing {1, 4, 6}: weights are the softmax of those unbiased logits
    b = torch.zeros(8, device=DEV)
    b[[1, 4, 6]] = 1e4
    idx2, w2 = pkg.moe_route(x, wr, b, 3)
    torch.cuda.synchronize()
    logits = oracle.router_logits(layer.x, wl.F32, layer.w_router, 8)
    ref = oracle.softmax_of_set(logits, idx2.cpu().numpy())
    assert np.all(np.sort(idx2.cpu().numpy(), 1) == [1, 4, 6])
    np.testing.assert_allclose(w2.cpu().numpy(), ref, atol=2e-6)


def test_device_status_ok_after_forward():
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(17, T=32, d=256, E=8, k=2, F=128, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    t = upload_layer(layer, DEV)
    ws = torch.empty(pkg.moe_workspace_size(32, 256, 8, 2, 128, 1, 1), dtype=torch.uint8,
                     device=DEV)
    gpu_forward(layer, DEV, t=t, workspace=ws)
    assert pkg.moe_check(ws) == 0


# -------------------------------------------------- workload sizes (full)
FULL_CASES = [("tiny_fp32", None), ("zonos3_mini_decode", None), ("zonos2_decode", 1),
              ("zonos2_decode", 8), ("zonos2_decode", 64), ("zonos3_mini_prefill", None),
              ("zonos2_prefill_q8", None), ("zonos2_decode_q4", 1), ("zonos2_decode_q4", 8),
              ("zonos2_decode_q4", 64), ("zonos2_prefill_q4", None), ("zonos2_decode_q4k", 1),
              ("zonos2_decode_q4k", 8), ("zonos2_decode_q4k", 64), ("zonos2_prefill_q4k", None),
              ("zonos2_decode_q6k", 1), ("zonos2_decode_q6k", 8), ("zonos2_decode_q6k", 64),
              ("zonos2_prefill_q6k", None), ("zonos2_decode_q8", 1), ("zonos2_decode_q8", 8),
              ("zonos2_decode_q8", 64), ("zonos2_decode_fp8", 1), ("zonos2_decode_fp8", 8),
              ("zonos2_decode_fp8", 64), ("zonos2_prefill_fp8", None)]


@pytest.mark.parametrize("seed", [2, 7, 13])
@pytest.mark.parametrize("name,T", FULL_CASES)
def test_forward_workloads_full(name, T, seed):
    """Every workload at full size, in the launch configuration the benchmark
    times (path AUTO): the routing and grouping the layer's own kernels wrote
    (read back from its workspace) against the oracle -- indices exact beyond
    the 1e-3 margin, near ties resolved validly, weights within 2e-6, counts,
    offsets, permutation and inverse bit-exact -- and every output row within
    the tolerance."""
    if ("_q4" in name or "_q6" in name or "decode_q8" in name or "_fp8" in name) and seed == 13:
        pytest.skip("the 4-, 6- and 8-bit workloads run with two seeds")
    layer = wl.make_layer(wl.WORKLOADS[name], seed=seed, T=T)
    out, r = gpu_forward_views(layer, DEV, path=0)
    check_routing_views(r, layer)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("name", ["zonos3_mini_prefill", "zonos2_prefill_q8", "zonos2_prefill_q4",
                                  "zonos2_prefill_q4k"])
def test_forward_prefill_workloads_on_decode_path(name):
    """The prefill workloads at full size through the decode path (CUDA-core
    kernels at these row counts): grouping and every output row."""
    layer = wl.make_layer(wl.WORKLOADS[name], seed=3)
    out, r = gpu_forward_views(layer, DEV, path=DECODE)
    check_routing_views(r, layer)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("name", ["zonos3_mini_decode", "zonos2_decode", "zonos3_mini_prefill",
                                  "zonos2_prefill_q8", "zonos2_decode_q4", "zonos2_prefill_q4",
                                  "zonos2_decode_q4k", "zonos2_prefill_q4k", "zonos2_decode_fp8",
                                  "zonos2_prefill_fp8"])
def test_graph_replay_equals_direct_launch(name):
    """The benchmark times CUDA-graph replays of the layer (warm-up launches on a
    side stream, capture on that stream, replay): at full size, a replay writes
    the same bits as a direct launch of the same layer."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_layer(wl.WORKLOADS[name], seed=4)
    t = upload_layer(layer, DEV)
    ws = torch.empty(pkg.moe_workspace_size(layer.T, layer.d, layer.E, layer.k, layer.F,
                                            layer.act_dtype, layer.w_dtype),
                     dtype=torch.uint8, device=DEV)
    direct = torch.empty((layer.T, layer.d), dtype=torch.float32, device=DEV)
    replay = torch.empty_like(direct)
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            gpu_forward(layer, DEV, t=t, out=direct, workspace=ws)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gpu_forward(layer, DEV, t=t, out=replay, workspace=ws)
    replay.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert torch.equal(direct, replay)
    assert pkg.moe_check(ws) == 0


# ------------------------------------------- tensor-core (prefill) path
PREFILL_SMALL = [
    # (T, d, E, k, F): ragged groups, tiles crossing expert boundaries, empty experts
    (130, 256, 2, 1, 128),
    (300, 256, 4, 2, 128),
    (1000, 512, 8, 2, 256),
    (2048, 256, 16, 1, 384),
    (520, 1024, 64, 2, 512),
    (777, 2048, 16, 1, 256),
    (600, 256, 4, 1, 1024),     # k == 1 (plain stores), long F: 16 k-blocks per down tile
    (700, 256, 256, 8, 128),    # the largest E and k: 5600 rows over 256 small groups
]


@pytest.mark.parametrize("wdt", [wl.BF16, wl.Q8_0, wl.Q4_A64])
@pytest.mark.parametrize("T,d,E,k,F", PREFILL_SMALL)
def test_forward_prefill_small_matches_oracle(T, d, E, k, F, wdt):
    layer = wl.make_custom_layer(21, T=T, d=d, E=E, k=k, F=F, act_dtype=wl.BF16,
                                 w_dtype=wdt, bias_sd=0.5)
    out, r = gpu_forward_views(layer, DEV, path=PREFILL)
    check_routing_views(r, layer)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("wdt", [wl.Q4_K, wl.Q6_K, wl.FP8])
@pytest.mark.parametrize("T,d,E,k,F", [c for c in PREFILL_SMALL if c[1] % 256 == 0 and c[4] % 256 == 0])
def test_forward_prefill_small_q4_k_matches_oracle(T, d, E, k, F, wdt):
    """Q4_K, Q6_K and fp8 experts on the grouped GEMMs (the shapes above with
    whole 256-value super-blocks along d and F)."""
    layer = wl.make_custom_layer(21, T=T, d=d, E=E, k=k, F=F, act_dtype=wl.BF16,
                                 w_dtype=wdt, bias_sd=0.5)
    out, r = gpu_forward_views(layer, DEV, path=PREFILL)
    check_routing_views(r, layer)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


def test_prefill_one_expert_many_tiles():
    """Every token to experts 3 and 5: 1100 rows per group, a ragged last tile."""
    layer = wl.make_custom_layer(22, T=1100, d=256, E=8, k=2, F=128, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    layer.bias[:] = 0
    layer.bias[3] = 100.0
    layer.bias[5] = 50.0
    out, r = gpu_forward_views(layer, DEV, path=PREFILL)
    check_routing_views(r, layer)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    assert np.all(idx_ref == [3, 5])
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("wdt", [wl.BF16, wl.Q8_0, wl.Q4_A64, wl.Q4_K, wl.Q6_K, wl.FP8])
def test_prefill_and_decode_paths_agree(wdt):
    layer = wl.make_custom_layer(23, T=640, d=512, E=8, k=2, F=256, act_dtype=wl.BF16,
                                 w_dtype=wdt)
    t = upload_layer(layer, DEV)
    a = gpu_forward(layer, DEV, path=SIMT, t=t).cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(a ** 2))
    for path in ((PREFILL,) if wdt in (wl.Q8_0, wl.Q6_K) else (DECODE, PREFILL)):   # (fp8: both)
        b = gpu_forward(layer, DEV, path=path, t=t).cpu().numpy().astype(np.float64)
        assert np.abs(a - b).max() <= 2e-2 * rms


@pytest.mark.parametrize("T,k", [(1, 1), (8, 1), (64, 1), (33, 2), (128, 2), (300, 4)])
def test_decode_tc_deterministic_and_equivariant(T, k):
    layer = wl.make_custom_layer(25, T=T, d=512, E=16, k=k, F=384, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16, bias_sd=0.5)
    t = upload_layer(layer, DEV)
    a = gpu_forward(layer, DEV, path=DECODE, t=t).cpu().numpy()
    b = gpu_forward(layer, DEV, path=DECODE, t=t).cpu().numpy()
    assert np.array_equal(a, b)
    perm = np.random.default_rng(2).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, path=DECODE, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])
    _, r = gpu_forward_views(layer, DEV, path=DECODE, t=t)
    check_routing_views(r, layer)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(a, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("T,d,E,k,F", [
    (2, 1024, 8, 1, 1024),   # clusters of 8 CTAs for both kernels (16 k-blocks, 16 units)
    (3, 512, 8, 2, 512),     # clusters of 4; k = 2: two additions onto the zeroed output
    (5, 256, 16, 2, 256),    # clusters of 2
    (1, 2048, 16, 1, 2816),  # the ZONOS2 shape: 22 gate/up and 16 down units, clusters of 8
    (24, 512, 4, 2, 256),    # 48 rows: chunks of 16 rows, several per expert
])
@pytest.mark.parametrize("wdt", [wl.BF16, wl.Q4_A64, wl.Q4_K, wl.FP8])
def test_decode_cluster_mode_deterministic_equivariant_and_matches_oracle(T, d, E, k, F, wdt):
    """Small decode batches run the tensor-core decode kernels in cluster
    mode: the K splits of a unit are reduced in shared memory across the
    cluster, in rank order.  Two runs give the same bits, permuting the
    tokens permutes the output rows bit for bit, and the result matches the
    oracle (bf16, affine 4-bit, Q4_K and fp8 weights: fp8 row scales act on
    each split's sums before the reduction)."""
    layer = wl.make_custom_layer(30, T=T, d=d, E=E, k=k, F=F, act_dtype=wl.BF16, w_dtype=wdt,
                                 bias_sd=0.5)
    t = upload_layer(layer, DEV)
    a, r = gpu_forward_views(layer, DEV, path=DECODE, t=t)
    b, _ = gpu_forward_views(layer, DEV, path=DECODE, t=t)
    assert np.array_equal(a, b)
    perm = np.random.default_rng(8).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, path=DECODE, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])
    check_routing_views(r, layer)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(a, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


@pytest.mark.parametrize("wdt", [wl.BF16, wl.Q8_0, wl.Q4_A64, wl.FP8])
@pytest.mark.parametrize("k,F", [(2, 128), (1, 1024)])   # (1, 1024): long K in the down GEMM
def test_prefill_deterministic_and_equivariant(wdt, k, F):
    layer = wl.make_custom_layer(24, T=512, d=256, E=8, k=k, F=F, act_dtype=wl.BF16,
                                 w_dtype=wdt)
    t = upload_layer(layer, DEV)
    a = gpu_forward(layer, DEV, path=PREFILL, t=t).cpu().numpy()
    b = gpu_forward(layer, DEV, path=PREFILL, t=t).cpu().numpy()
    assert np.array_equal(a, b)
    perm = np.random.default_rng(1).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, path=PREFILL, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])


# ---------------------------------------- other scoring modes (next row f1)
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("act,T", [(wl.F32, 37), (wl.BF16, 200), (wl.BF16, 700)])
def test_route_scored_matches_oracle(mode, act, T):
    """CUDA-core router (fp32, bf16 below 512 tokens) and tensor-core router
    (bf16, 512 tokens and more) in softmax / sigmoid-before-rank mode."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(31, T=T, d=256, E=24, k=3, F=128, act_dtype=act, w_dtype=act,
                                 bias_sd=0.05)
    x, wr, b = to_dev(layer.x, DEV), to_dev(layer.w_router, DEV), to_dev(layer.bias, DEV)
    idx, w = pkg.moe_route(x, wr, b, layer.k, scoring=mode)
    torch.cuda.synchronize()
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    idx_ref, w_ref, margin = oracle.route_scored(logits, layer.bias, layer.k, mode)
    ok = compare_routing(idx.cpu().numpy(), w.cpu().numpy(), idx_ref, w_ref, margin, layer.k, mode)
    assert ok.mean() > 0.5


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("path,T,wdt", [(DECODE, 40, wl.BF16), (SIMT, 40, wl.BF16),
                                        (PREFILL, 600, wl.BF16), (PREFILL, 600, wl.Q8_0)])
def test_forward_scored_matches_oracle(mode, path, T, wdt):
    """Whole layer in softmax / sigmoid-before-rank mode on the clustered
    decode router, the CUDA-core router and the tensor-core prefill router."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(32, T=T, d=256, E=16, k=2, F=256, act_dtype=wl.BF16,
                                 w_dtype=wdt, bias_sd=0.05)
    out, r = gpu_forward_views(layer, DEV, path=path, scoring=mode)
    check_routing_views(r, layer, mode=mode)
    ref, idx_ref, w_ref, margin = oracle.moe_forward(layer, mode=mode)
    check_output(out, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"], mode=mode)


# ---------------------------------------- dense SwiGLU layer (next row f2)
@pytest.mark.parametrize("act,wdt,T,path", [
    (wl.BF16, wl.BF16, 5, DECODE), (wl.BF16, wl.BF16, 5, SIMT), (wl.F32, wl.F32, 37, SIMT),
    (wl.BF16, wl.Q8_0, 9, SIMT), (wl.BF16, wl.BF16, 600, PREFILL), (wl.BF16, wl.Q8_0, 600, PREFILL),
    (wl.BF16, wl.BF16, 700, 0), (wl.BF16, wl.Q4_A64, 40, DECODE)])
def test_ffn_dense_matches_oracle(act, wdt, T, path):
    """moe_ffn_dense against the oracle's one-expert layer, and bit for bit
    against moe_forward with E = 1, k = 1 (same expert kernels; only the
    routing step differs)."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    layer = wl.make_custom_layer(33, T=T, d=256, E=1, k=1, F=256, act_dtype=act, w_dtype=wdt)
    t = upload_layer(layer, DEV)
    out = pkg.moe_ffn_dense(t["x"], t["w_gate"], t["w_up"], t["w_down"], F=layer.F,
                            w_dtype=layer.w_dtype, path=path).cpu().numpy()
    via_moe = gpu_forward(layer, DEV, path=path, t=t).cpu().numpy()
    assert np.array_equal(out, via_moe)
    # the dense call's own grouping: every token to expert 0 with weight 1, identity order
    ws = torch.empty(max(pkg.moe_workspace_size(T, 256, 1, 1, 256, act, wdt), 256),
                     dtype=torch.uint8, device=DEV)
    pkg.moe_ffn_dense(t["x"], t["w_gate"], t["w_up"], t["w_down"], F=layer.F,
                      w_dtype=layer.w_dtype, path=path, workspace=ws)
    torch.cuda.synchronize()
    r = {n: v.cpu().numpy() for n, v in pkg.read_routing(ws, T, 256, 1, 1, 256, act, wdt).items()}
    assert np.all(r["topk_idx"] == 0) and np.all(r["topk_w"] == 1.0) and np.all(r["perm_w"] == 1.0)
    assert r["counts"].tolist() == [T] and r["offsets"].tolist() == [0, T]
    assert np.array_equal(r["perm_tok"], np.arange(T)) and np.array_equal(r["inv"], np.arange(T))
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(out, layer, ref, idx_ref, margin)


# ------------------------------------------------ k > 2: reproducible everywhere
@pytest.mark.parametrize("k", [4, 8])
@pytest.mark.parametrize("path,T,act,wdt", [
    (DECODE, 64, wl.BF16, wl.BF16),     # tensor-core decode kernels (split-K + combine)
    (SIMT, 64, wl.BF16, wl.BF16),       # CUDA-core decode kernels
    (SIMT, 40, wl.F32, wl.F32),
    (SIMT, 40, wl.BF16, wl.Q8_0),
    (PREFILL, 600, wl.BF16, wl.BF16),   # grouped GEMMs
    (PREFILL, 600, wl.BF16, wl.Q8_0),
    (DECODE, 64, wl.BF16, wl.FP8),      # fp8: row scales before the slot-order combine
    (SIMT, 40, wl.BF16, wl.FP8),
    (PREFILL, 600, wl.BF16, wl.FP8),
])
def test_k_above_two_reproducible_and_equivariant(path, T, act, wdt, k):
    """With k > 2 every path adds a token's k expert outputs in slot order (no
    atomics): two runs give the same bits, permuting the tokens permutes the
    output rows bit for bit, and the result matches the oracle."""
    layer = wl.make_custom_layer(26, T=T, d=256, E=16, k=k, F=128, act_dtype=act, w_dtype=wdt,
                                 bias_sd=0.5)
    t = upload_layer(layer, DEV)
    a, r = gpu_forward_views(layer, DEV, path=path, t=t)
    b, _ = gpu_forward_views(layer, DEV, path=path, t=t)
    assert np.array_equal(a, b)
    perm = np.random.default_rng(3).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, path=path, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])
    check_routing_views(r, layer)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_output(a, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])


# ------------------- fp16 operands of the Q8_0 GEMMs and the 4-bit decode kernels
@pytest.mark.parametrize("path,T,wdt,E,F", [
    (PREFILL, 300, wl.Q8_0, 8, 256), (SIMT, 40, wl.Q8_0, 8, 256), (0, 600, wl.Q8_0, 8, 256),
    (DECODE, 40, wl.Q4_A64, 8, 256),      # split-K gate/up + SwiGLU reduction
    (DECODE, 128, wl.Q4_A64, 64, 512),    # whole-K gate/up writing h itself
    (DECODE, 300, wl.Q4_A64, 8, 256),     # rows grouped by the scatter kernel
    (PREFILL, 600, wl.Q4_A64, 8, 256),    # 4-bit grouped GEMMs
    (DECODE, 40, wl.Q4_K, 8, 256), (PREFILL, 600, wl.Q4_K, 8, 256),
    (DECODE, 40, wl.Q8_0, 8, 256), (DECODE, 128, wl.Q6_K, 64, 512),   # 8-bit planes, decode
    (PREFILL, 600, wl.Q6_K, 8, 256),    # Q6_K grouped GEMMs: scales per 16 values
    (DECODE, 40, wl.FP8, 8, 256), (DECODE, 128, wl.FP8, 64, 512),   # fp8: row scales on the sums
    (PREFILL, 600, wl.FP8, 8, 256)])
def test_fp16_operands_large_activations(path, T, wdt, E, F):
    """The Q8_0 grouped GEMMs and the 4-bit tensor-core decode kernels
    multiply fp16 operands.  Token rows whose magnitudes span 1e-2 .. 1e5 (h
    far beyond fp16's 65504 for the large ones) match the oracle: each fp16
    row is the bf16 row times an exact power of two, undone exactly in the
    epilogues."""
    layer = wl.make_custom_layer(27, T=T, d=256, E=E, k=2, F=F, act_dtype=wl.BF16,
                                 w_dtype=wdt, bias_sd=0.3)
    mag = 10.0 ** np.random.default_rng(5).uniform(-2, 5, size=T)
    mag[:4] = [1e5, 2e-2, 1.0, 7e4]
    x = wl.bf16_bits_to_f32(layer.x) * mag[:, None].astype(np.float32)
    layer.x = wl.f32_to_bf16_bits(x)
    out, r = gpu_forward_views(layer, DEV, path=path)
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    assert np.abs(ref).max() > 65504.0 ** 2 * 1e-3     # h and out far beyond fp16's range
    # logits of 1e5-magnitude rows carry the router's fp32 accumulation error
    # (~1e-7 of |logit| ~ 1e4): their weights agree to ~1e-5, not 2e-6
    check_routing_views(r, layer, w_atol=5e-5)
    # per decade of row magnitude: out grows like mag^2, so the largest rows
    # dominate any wider bin's RMS and each row is held to the tolerance of
    # rows of its own magnitude
    decade = np.clip(np.floor(np.log10(mag)), -2, 4)    # mag = 1e5 joins [1e4, 1e5)
    for lo in np.unique(decade):
        rows = decade == lo
        if rows.any():
            sub_rows = np.where(rows)[0]
            from helpers import sub_layer
            sub = sub_layer(layer, sub_rows)
            check_output(out[sub_rows], sub, ref[sub_rows], idx_ref[sub_rows], margin[sub_rows],
                         idx_gpu=r["topk_idx"][sub_rows])


@pytest.mark.parametrize("wdt,path,T,E,k,F", [
    (wl.Q8_0, PREFILL, 256, 4, 1, 128),
    (wl.Q4_A64, DECODE, 256, 4, 1, 128),     # 4-bit: SwiGLU reduction kernel
    (wl.Q4_A64, DECODE, 128, 64, 2, 512),    # 4-bit: whole-K gate/up epilogue
    (wl.Q4_A64, PREFILL, 256, 4, 1, 128),    # 4-bit grouped GEMMs
    (wl.Q4_K, DECODE, 256, 4, 1, 256),
    (wl.Q4_K, PREFILL, 256, 4, 1, 256),
    (wl.Q6_K, PREFILL, 256, 4, 1, 256),
    (wl.Q8_0, DECODE, 256, 4, 1, 256), (wl.Q6_K, DECODE, 128, 64, 2, 512),
    (wl.FP8, DECODE, 256, 4, 1, 128), (wl.FP8, PREFILL, 256, 4, 1, 128)])
def test_fp16_h_beyond_range_is_reported(wdt, path, T, E, k, F):
    """Expert weights large enough that h leaves fp16's range even for
    normalised rows: the call reports MOE_ERR_DEVICE_CHECK instead of
    returning infinities silently."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    d = 256
    layer = wl.make_custom_layer(28, T=T, d=d, E=E, k=k, F=F, act_dtype=wl.BF16,
                                 w_dtype=wl.BF16)
    rng = np.random.default_rng(6)
    big = lambda *s: (rng.standard_normal(s) * 4e3).astype(np.float32)
    quant = {wl.Q8_0: wl.q8_0_quantize, wl.Q4_A64: wl.q4_a64_quantize,
             wl.Q4_K: wl.q4_k_quantize, wl.Q6_K: wl.q6_k_quantize, wl.FP8: wl.fp8_quantize}[wdt]
    layer.w_dtype = wdt
    layer.w_gate = quant(big(E, F, d))
    layer.w_up = quant(big(E, F, d))
    layer.w_down = quant(big(E, d, F) * 1e-3)
    t = upload_layer(layer, DEV)
    ws = torch.empty(pkg.moe_workspace_size(T, d, E, k, F, 1, wdt), dtype=torch.uint8,
                     device=DEV)
    gpu_forward(layer, DEV, path=path, t=t, workspace=ws)
    torch.cuda.synchronize()
    word = ctypes_check(pkg, ws)
    assert word == 6, word            # MOE_ERR_DEVICE_CHECK


def ctypes_check(pkg, ws):
    import ctypes
    L = pkg.load_library()
    w = ctypes.c_uint32(0)
    return L.moe_check(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(w),
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("wdt,F", [(wl.Q4_A64, 384), (wl.Q4_K, 512), (wl.Q8_0, 384), (wl.Q6_K, 512),
                                   (wl.FP8, 384)])
@pytest.mark.parametrize("T,k", [(1, 1), (8, 1), (64, 1), (40, 2), (200, 4)])
def test_q4_tensor_core_decode_reproducible_and_close_to_cuda_core(T, k, wdt, F):
    """Affine 4-bit, Q4_K, Q8_0, Q6_K and fp8 experts on the tensor-core decode
    kernels (converter warps write the fp16 weights into tensor memory):
    bitwise reproducible, token-permutation equivariant, within tolerance of
    the oracle and of the CUDA-core kernels."""
    layer = wl.make_custom_layer(29, T=T, d=512, E=16, k=k, F=F, act_dtype=wl.BF16,
                                 w_dtype=wdt, bias_sd=0.5)
    t = upload_layer(layer, DEV)
    a, r = gpu_forward_views(layer, DEV, path=DECODE, t=t)
    b, _ = gpu_forward_views(layer, DEV, path=DECODE, t=t)
    assert np.array_equal(a, b)
    perm = np.random.default_rng(4).permutation(layer.T)
    t2 = dict(t, x=t["x"][torch.from_numpy(perm).to(DEV)].contiguous())
    c = gpu_forward(layer, DEV, path=DECODE, t=t2).cpu().numpy()
    assert np.array_equal(c, a[perm])
    ref, idx_ref, _, margin = oracle.moe_forward(layer)
    check_routing_views(r, layer)
    check_output(a, layer, ref, idx_ref, margin, idx_gpu=r["topk_idx"])
    simt, _ = gpu_forward_views(layer, DEV, path=SIMT, t=t)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(a.astype(np.float64) - simt).max() <= 2e-2 * rms


@pytest.mark.parametrize("rows,cols", [(130, 128), (256, 192), (1, 64)])
def test_q4_pack_tile_layout(rows, cols):
    """moe_pack_q4_a64's output, byte for byte, against the tile layout its
    header states, built here from the 36-byte blocks with numpy: tile
    (row // 128, group) at ((row // 128) * groups + group) * 4608 holds the
    128 rows' 32 code bytes (each 32-bit word: values 0, 2, 4, 6 in nibbles
    0-3, values 1, 3, 5, 7 in nibbles 4-7), then their fp16 scales, then their
    biases; rows past the last are zero."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rng = np.random.default_rng(rows + cols)
    w = rng.standard_normal((rows, cols)).astype(np.float32)
    blocks = wl.q4_a64_quantize(w)                     # [rows, cols/64, 36]
    packed = pkg.moe_pack_q4_a64(torch.from_numpy(blocks.reshape(-1).copy()).to(DEV), rows, cols)
    got = packed.cpu().numpy()
    G, RT = cols // 64, (rows + 127) // 128
    want = np.zeros(RT * G * 4608, dtype=np.uint8)
    for r in range(rows):
        for g in range(G):
            t = ((r // 128) * G + g) * 4608
            rr = r % 128
            codes = blocks[r, g, 4:].astype(np.uint32).reshape(8, 4)   # 4 bytes per word
            lo = codes & 15                                           # values 0, 2, 4, 6
            hi = codes >> 4                                           # values 1, 3, 5, 7
            words = (lo << np.array([0, 4, 8, 12], dtype=np.uint32)).sum(1) | \
                ((hi << np.array([16, 20, 24, 28], dtype=np.uint32)).sum(1))
            want[t + rr * 32:t + rr * 32 + 32] = words.astype("<u4").view(np.uint8)
            want[t + 4096 + 2 * rr:t + 4098 + 2 * rr] = blocks[r, g, 0:2]
            want[t + 4352 + 2 * rr:t + 4354 + 2 * rr] = blocks[r, g, 2:4]
    assert got.shape == want.shape and np.array_equal(got, want)


def q4_k_fields(blk):
    """(d, dmin, sc[8], m[8]) of one 144-byte Q4_K super-block, decoded here
    with numpy from the six-bit field layout moe.h states."""
    d = float(np.frombuffer(blk[0:2].tobytes(), "<f2")[0])
    dmin = float(np.frombuffer(blk[2:4].tobytes(), "<f2")[0])
    s = blk[4:16].astype(np.int64)
    sc, m = np.zeros(8, np.int64), np.zeros(8, np.int64)
    for j in range(8):
        if j < 4:
            sc[j], m[j] = s[j] & 63, s[j + 4] & 63
        else:
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
            m[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
    return d, dmin, sc, m


@pytest.mark.parametrize("rows,cols", [(130, 256), (256, 512), (1, 256)])
def test_q4_k_pack_tile_layout(rows, cols):
    """moe_pack_q4_k's output, byte for byte, against the tile layout its
    header states, built here from the 144-byte super-blocks with numpy: tile
    (row // 128, kb) at ((row // 128) * (cols / 64) + kb) * 5120 holds the 64
    values 64 kb .. 64 kb + 63 of its 128 rows as code words (the 4-bit words
    of the affine 4-bit tiles), then fp16 scales [2][128], then fp16 biases
    [2][128]: group g is sub-block j = 2 (kb % 4) + g of super-block kb // 4,
    scale = fp16(d * sc[j]), bias = fp16(8 d sc[j] - dmin m[j]) (the value at
    code 8); rows past the last are zero."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rng = np.random.default_rng(rows + cols + 1)
    w = (rng.standard_normal((rows, cols)) * rng.uniform(0.1, 3.0, (rows, 1))).astype(np.float32)
    blocks = wl.q4_k_quantize(w)                       # [rows, cols/256, 144]
    n = pkg.moe_q4_k_packed_size(rows, cols)
    packed = pkg.moe_pack_q4_k(torch.from_numpy(blocks.reshape(-1).copy()).to(DEV), rows, cols)
    got = packed.cpu().numpy()[:n]
    G, RT = cols // 64, (rows + 127) // 128
    want = np.zeros(RT * G * 5120, dtype=np.uint8)
    shifts_lo = np.array([0, 4, 8, 12], dtype=np.uint32)
    shifts_hi = np.array([16, 20, 24, 28], dtype=np.uint32)
    for r in range(rows):
        for kb in range(G):
            blk = blocks[r, kb // 4]
            dd, dmin, sc, m = q4_k_fields(blk)
            run = blk[16 + 32 * (kb % 4):48 + 32 * (kb % 4)].astype(np.uint32)
            vals = np.concatenate([run & 15, run >> 4])        # the 64 codes in value order
            t = ((r // 128) * G + kb) * 5120
            rr = r % 128
            v = vals.reshape(8, 8)                               # word i: values 8i .. 8i+7
            words = (v[:, 0::2] << shifts_lo).sum(1) | (v[:, 1::2] << shifts_hi).sum(1)
            want[t + rr * 32:t + rr * 32 + 32] = words.astype("<u4").view(np.uint8)
            for g in range(2):
                j = 2 * (kb % 4) + g
                s32 = np.float32(dd) * np.float32(sc[j])             # exact in fp32
                scale = np.float16(s32)
                bias = np.float16(np.float32(8) * s32 - np.float32(dmin) * np.float32(m[j]))
                want[t + 4096 + 256 * g + 2 * rr:t + 4098 + 256 * g + 2 * rr] = \
                    np.array([scale]).view(np.uint8)
                want[t + 4608 + 256 * g + 2 * rr:t + 4610 + 256 * g + 2 * rr] = \
                    np.array([bias]).view(np.uint8)
    assert got.shape == want.shape and np.array_equal(got, want)


@pytest.mark.parametrize("rows,cols", [(130, 256), (3, 512)])
def test_q6_k_pack_planes(rows, cols):
    """moe_pack_q6_k's output, byte for byte, against the planes its header
    states, built here with numpy from the 210-byte super-blocks: the int8
    plane [rows, cols] holds q - 32 of every value (low nibble from ql, top
    bits from qh), and the fp16 plane [cols/16, rows] at align256(rows*cols)
    holds fp16(d * scales[j]) of 16-value group j."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rng = np.random.default_rng(rows * 7 + cols)
    w = (rng.standard_normal((rows, cols)) * rng.uniform(0.1, 3.0, (rows, 1))).astype(np.float32)
    blocks = wl.q6_k_quantize(w)                       # [rows, cols/256, 210]
    n = pkg.moe_q6_k_packed_size(rows, cols)
    got = pkg.moe_pack_q6_k(torch.from_numpy(blocks.reshape(-1).copy()).to(DEV), rows, cols).cpu().numpy()[:n]
    q = np.zeros((rows, cols), np.int8)
    scales = np.zeros((cols // 16, rows), np.float16)
    for r in range(rows):
        for sb in range(cols // 256):
            blk = blocks[r, sb]
            d = np.float32(blk[208:210].copy().view(np.float16)[0])
            sc = blk[192:208].copy().view(np.int8)
            for v in range(256):
                h, g, l = v // 128, (v % 128) // 32, v % 32
                lo_byte = int(blk[64 * h + l + 32 * (g % 2)])
                lo = (lo_byte & 15) if g < 2 else (lo_byte >> 4)
                hi = (int(blk[128 + 32 * h + l]) >> (2 * g)) & 3
                q[r, 256 * sb + v] = (lo | (hi << 4)) - 32
            for j in range(16):
                scales[16 * sb + j, r] = np.float16(d * np.float32(sc[j]))
    off = (rows * cols + 255) // 256 * 256
    assert n == off + scales.size * 2
    assert np.array_equal(got[:rows * cols], q.reshape(-1).view(np.uint8))
    assert np.array_equal(got[off:n], scales.reshape(-1).view(np.uint8))


@pytest.mark.parametrize("rows,cols", [(130, 128), (3, 2048), (1, 8)])
def test_fp8_pack_planes(rows, cols):
    """moe_pack_fp8's output, byte for byte, against the layout its header
    states, built here with numpy from the rows {fp32 scale, E4M3 codes}: the
    E4M3 plane [rows, cols], then at align256(rows*cols) the fp32 scales."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rng = np.random.default_rng(rows + cols)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    src = wl.fp8_quantize(w)                       # [rows, 4 + cols]
    n = pkg.moe_fp8_packed_size(rows, cols)
    plane_end = (rows * cols + 255) // 256 * 256
    assert n == plane_end + 4 * rows
    got = pkg.moe_pack_fp8(torch.from_numpy(src.reshape(-1).copy()).to(DEV), rows, cols).cpu().numpy()[:n]
    assert np.array_equal(got[:rows * cols], src[:, 4:].reshape(-1))
    assert np.array_equal(got[plane_end:plane_end + 4 * rows].view(np.float32),
                          src[:, 0:4].copy().view(np.float32)[:, 0])
