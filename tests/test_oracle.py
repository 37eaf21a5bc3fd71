"""Pins of the CPU oracle against what the definition and mathematics fix.

Definition: SelectedSoftmax routing ("New Community Model: ZONOS3-Mini
(Zyphra) - #1271", §Framework change) feeding SwiGLU experts ("zonos2.cpp
internals", §Recommended: F16 spine + K-quant experts, expert stacks
ffn_{gate,up,down}_exps).  Each test is chosen so that a plausible slip in the
oracle -- biased logits in the softmax, a wrong tie-break, a transposed weight,
a dropped SiLU factor, an off-by-one in the scan -- fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "selected_softmax_worked.txt")


def _golden():
    cases = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "case":
            cases.setdefault(parts[1], {})[parts[2]] = [float(v) for v in parts[3:]]
        elif parts[0] == "ffn":
            cases["ffn"] = [float(v) for v in parts[2:]]
    return cases


# ------------------------------------------------ independent numpy helpers
def decode(a, dtype):
    """Storage -> float64, written independently of the C oracle."""
    if dtype == wl.F32:
        return np.asarray(a, np.float32).astype(np.float64)
    if dtype == wl.BF16:
        return wl.bf16_bits_to_f32(a).astype(np.float64)
    blocks = np.asarray(a, np.uint8)
    if dtype == wl.FP8:
        # rows {fp32 scale, E4M3 codes}: the codes through torch's float8_e4m3fn
        import torch
        scale = blocks[..., 0:4].copy().view(np.float32)[..., 0].astype(np.float64)
        codes = torch.from_numpy(np.ascontiguousarray(blocks[..., 4:])).view(torch.float8_e4m3fn)
        return scale[..., None] * codes.float().numpy().astype(np.float64)
    if dtype == wl.Q6_K:
        # 256 values per 210 bytes: ql[128] low 4 bits, qh[64] top 2 bits,
        # int8 scales[16] (one per 16 values), fp16 d; code q, value d*sc*(q-32).
        # Written per value from the layout: v = 128h + 32g + l.
        d6 = blocks[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
        sc6 = blocks[..., 192:208].copy().view(np.int8).astype(np.float64)
        w = np.empty(blocks.shape[:-1] + (256,), np.float64)
        for v in range(256):
            h, g, l = v // 128, (v % 128) // 32, v % 32
            lo_byte = blocks[..., 64 * h + l + 32 * (g % 2)].astype(np.int64)
            lo = (lo_byte & 15) if g < 2 else (lo_byte >> 4)
            hi = (blocks[..., 128 + 32 * h + l].astype(np.int64) >> (2 * g)) & 3
            w[..., v] = d6 * sc6[..., v // 16] * ((lo + 16 * hi) - 32)
        return w.reshape(w.shape[:-2] + (w.shape[-2] * w.shape[-1],))
    scale = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    if dtype == wl.Q4_K:
        # 256 values per 144 bytes: d, dmin, 12 bytes of 6-bit (scale, min)
        # pairs, 4 runs of 32 code bytes (low nibbles: sub-block 2c, high: 2c+1)
        dmin = blocks[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
        s = blocks[..., 4:16].astype(np.int64)
        w = np.empty(blocks.shape[:-1] + (256,), np.float64)
        for j in range(8):
            if j < 4:
                sc, mn = s[..., j] & 63, s[..., j + 4] & 63
            else:
                sc = (s[..., j + 4] & 15) + 16 * (s[..., j - 4] >> 6)
                mn = (s[..., j + 4] >> 4) + 16 * (s[..., j] >> 6)
            run = blocks[..., 16 + 32 * (j // 2):48 + 32 * (j // 2)].astype(np.int64)
            q = (run >> 4) if j % 2 else (run & 15)
            w[..., 32 * j:32 * j + 32] = scale[..., None] * sc[..., None] * q - dmin[..., None] * mn[..., None]
        return w.reshape(w.shape[:-2] + (w.shape[-2] * w.shape[-1],))
    if dtype == wl.Q4_A64:   # {scale, bias, 32 bytes: value 2j low nibble, 2j+1 high}
        bias = blocks[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
        codes = blocks[..., 4:]
        q = np.empty(codes.shape[:-1] + (64,), np.float64)
        q[..., 0::2] = codes & 15
        q[..., 1::2] = codes >> 4
        w = q * scale[..., None] + bias[..., None]
        return w.reshape(w.shape[:-2] + (w.shape[-2] * w.shape[-1],))
    q = blocks[..., 2:].copy().view(np.int8).astype(np.float64)
    w = q * scale[..., None]
    return w.reshape(w.shape[:-2] + (w.shape[-2] * w.shape[-1],))


def brute_force_dense(layer):
    """All experts on every token, then a brute-force top-k mask.

    The ranking uses Python's sort on (-score, expert) tuples, so ties go to
    the lower expert index; weights are exp(l - max) over the mask.
    """
    x = decode(layer.x, layer.act_dtype)
    wr = decode(layer.w_router, layer.act_dtype)
    wg = decode(layer.w_gate, layer.w_dtype)
    wu = decode(layer.w_up, layer.w_dtype)
    wd = decode(layer.w_down, layer.w_dtype)
    b = np.asarray(layer.bias, np.float64)
    T, E, k = x.shape[0], layer.E, layer.k
    logits = np.array([[sum(x[t, i] * wr[e, i] for i in range(x.shape[1])) for e in range(E)]
                       for t in range(T)])
    # dense: every expert for every token, [E, T, d]
    g = np.einsum("efi,ti->etf", wg, x)
    u = np.einsum("efi,ti->etf", wu, x)
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    y = np.einsum("eif,etf->eti", wd, h)
    out = np.zeros_like(x)
    sel_all = []
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-(logits[t, e] + b[e]), e))
        sel = order[:k]
        sel_all.append(sel)
        m = max(logits[t, e] for e in sel)
        z = sum(math.exp(logits[t, e] - m) for e in sel)
        for e in sel:
            out[t] += math.exp(logits[t, e] - m) / z * y[e, t]
    return out, np.array(sel_all, dtype=np.int32), logits


def tiny_layer(seed=0, act=wl.F32, wdt=wl.F32, T=8, d=64, E=8, k=2, F=128, bias_sd=0.1):
    return wl.make_custom_layer(seed, T, d, E, k, F, act, wdt, bias_sd=bias_sd)


# ---------------------------------------------------------------- the pins
def test_golden_worked_routing():
    gold = _golden()
    x = np.array([[1.0, 0.0]], np.float32)
    wr = np.array([[0.5, 0], [1, 0], [-1, 0], [2, 0]], np.float32)
    logits = oracle.router_logits(x, wl.F32, wr, 4)
    assert logits.tolist() == [[0.5, 1.0, -1.0, 2.0]]
    bias_a = np.array([3, 0, 0, 0], np.float32)
    for name, bias, k in (("A", bias_a, 2), ("B", None, 2), ("D", bias_a, 1)):
        idx, w, _ = oracle.selected_softmax(logits, bias, k)
        assert idx[0].tolist() == [int(v) for v in gold[name]["idx"]], name
        np.testing.assert_allclose(w[0], gold[name]["w"], rtol=1e-15, atol=0)
    tie = np.array([[1.0, 1.0, 0.0, 1.0]])
    idx, w, margin = oracle.selected_softmax(tie, None, 2)
    assert idx[0].tolist() == [int(v) for v in gold["C"]["idx"]]
    assert w[0].tolist() == gold["C"]["w"]
    assert margin[0] == 0.0


def test_golden_worked_ffn():
    gold = _golden()
    x = np.array([[1.0, 2.0]], np.float32)
    wg = np.array([[[1, 0], [0, -1]]], np.float32)
    wu = np.array([[[2, 0], [1, 1]]], np.float32)
    wd = np.array([[[1, 3], [5, 7]]], np.float32)
    out = oracle.expert_combine(x, wl.F32, np.array([[0]]), np.array([[1.0]]), wg, wu, wd,
                                wl.F32, 1, 2)
    np.testing.assert_allclose(out[0], gold["ffn"], rtol=1e-14, atol=0)


def test_k1_weight_is_exactly_one():
    layer = tiny_layer(k=1, E=16)
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    _, w, _ = oracle.selected_softmax(logits, layer.bias, 1)
    assert np.all(w == 1.0)


@pytest.mark.parametrize("k", [2, 3, 4, 8])
def test_weights_sum_to_one(k):
    rng = np.random.default_rng(k)
    logits = rng.standard_normal((64, 16)) * 3
    idx, w, _ = oracle.selected_softmax(logits, rng.standard_normal(16).astype(np.float32), k)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-15)
    assert np.all(w > 0)
    # each row's slots are distinct experts, in descending ranking score
    for t in range(64):
        assert len(set(idx[t].tolist())) == k


def test_bias_selects_but_never_weighs():
    rng = np.random.default_rng(3)
    T, E, k = 32, 12, 3
    logits = rng.standard_normal((T, E))
    idx0, w0, margin0 = oracle.selected_softmax(logits, None, k)
    # a bias too small to change any selection leaves weights bit-identical
    small = (rng.standard_normal(E) * 1e-9).astype(np.float32)
    ok = margin0 > 1e-6
    idx1, w1, _ = oracle.selected_softmax(logits, small, k)
    assert np.array_equal(idx1[ok], idx0[ok])
    assert np.array_equal(w1[ok], w0[ok])
    # a bias forcing set S = {1, 5, 7} gives weights = softmax of the S logits
    force = np.zeros(E, np.float32)
    force[[1, 5, 7]] = 1e6
    idx2, w2, _ = oracle.selected_softmax(logits, force, k)
    for t in range(T):
        assert sorted(idx2[t].tolist()) == [1, 5, 7]
        l = logits[t, idx2[t]]
        ref = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
        np.testing.assert_allclose(w2[t], ref, rtol=1e-14)


def test_softmax_of_set_pinned():
    """The set-weights helper (the weights of a fixed expert set, used to
    re-evaluate near-tie tokens with another set) against a library softmax
    (scipy) of the set's logits, bit for bit against the router's own weights
    for the set the router keeps, the two-expert closed form 1/(1+e^-delta),
    and exactly 1 for a single expert ("New Community Model: ZONOS3-Mini
    (Zyphra) - #1271", §Framework change: the kept experts are weighed by the
    softmax of their logits)."""
    from scipy.special import softmax
    rng = np.random.default_rng(44)
    T, E = 50, 16
    logits = rng.standard_normal((T, E)) * 3
    for k in (1, 2, 3, 8):
        # arbitrary sets in arbitrary slot order, not the router's
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        w = oracle.softmax_of_set(logits, idx)
        ref = softmax(np.take_along_axis(logits, idx, axis=1), axis=1)
        np.testing.assert_allclose(w, ref, rtol=1e-14, atol=0)
        if k == 1:
            assert np.all(w == 1.0)
        # for the router's own set: the router's weights, bit for bit
        bias = (rng.standard_normal(E) * 0.5).astype(np.float32)
        idx_r, w_r, _ = oracle.selected_softmax(logits, bias, k)
        assert np.array_equal(oracle.softmax_of_set(logits, idx_r), w_r)
    # two experts: w0 = 1 / (1 + exp(-(l0 - l1)))
    idx2 = np.tile(np.array([[3, 9]], np.int32), (T, 1))
    w2 = oracle.softmax_of_set(logits, idx2)
    delta = logits[:, 3] - logits[:, 9]
    np.testing.assert_allclose(w2[:, 0], 1.0 / (1.0 + np.exp(-delta)), rtol=1e-14)
    np.testing.assert_allclose(w2[:, 1], 1.0 / (1.0 + np.exp(delta)), rtol=1e-14)


def test_zero_bias_is_textbook_topk_softmax_renormalised():
    """bias = 0: softmax over all E, keep the top k, renormalise."""
    rng = np.random.default_rng(4)
    T, E, k = 40, 10, 4
    logits = rng.standard_normal((T, E)) * 2
    idx, w, _ = oracle.selected_softmax(logits, None, k)
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for t in range(T):
        top = np.argsort(-p[t], kind="stable")[:k]
        assert idx[t].tolist() == top.tolist()
        np.testing.assert_allclose(w[t], p[t, top] / p[t, top].sum(), rtol=1e-13)


def test_k_equals_e_is_dense_softmax_gating():
    layer = tiny_layer(seed=5, E=4, k=4, T=6, d=32, F=64, bias_sd=3.0)
    out, idx, w, margin = oracle.moe_forward(layer)
    assert np.all(np.isinf(margin))
    x = decode(layer.x, wl.F32)
    logits = x @ decode(layer.w_router, wl.F32).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    wg, wu, wd = (decode(a, wl.F32) for a in (layer.w_gate, layer.w_up, layer.w_down))
    ref = np.zeros_like(x)
    for e in range(4):
        g, u = x @ wg[e].T, x @ wu[e].T
        ref += p[:, e:e + 1] * ((g / (1 + np.exp(-g)) * u) @ wd[e].T)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("act,wdt", [(wl.F32, wl.F32), (wl.BF16, wl.BF16), (wl.BF16, wl.Q8_0),
                                     (wl.BF16, wl.Q4_A64), (wl.BF16, wl.Q4_K), (wl.BF16, wl.Q6_K),
                                     (wl.BF16, wl.FP8)])
@pytest.mark.parametrize("k", [1, 2, 3])
def test_matches_dense_brute_force(act, wdt, k):
    d, F = (256, 256) if wdt in (wl.Q4_K, wl.Q6_K) else (64, 96) if wdt != wl.Q4_A64 else (64, 128)
    layer = tiny_layer(seed=10 + k, act=act, wdt=wdt, T=5, d=d, E=6, k=k, F=F, bias_sd=0.3)
    out, idx, w, margin = oracle.moe_forward(layer)
    ref, sel, logits = brute_force_dense(layer)
    assert np.array_equal(idx, sel)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_identical_experts_give_one_ffn():
    layer = tiny_layer(seed=6, k=3, E=5)
    for name in ("w_gate", "w_up", "w_down"):
        a = getattr(layer, name)
        a[:] = a[0:1]
    out, idx, w, _ = oracle.moe_forward(layer)
    ref = oracle.expert_combine(layer.x, wl.F32, np.zeros((layer.T, 1), np.int32),
                                np.ones((layer.T, 1)), layer.w_gate, layer.w_up,
                                layer.w_down, wl.F32, layer.E, layer.F)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-14)


def test_zero_up_projection_gives_zero():
    layer = tiny_layer(seed=7)
    layer.w_up[:] = 0
    out, *_ = oracle.moe_forward(layer)
    assert np.all(out == 0.0)


def test_token_permutation_equivariance_bit_exact():
    layer = tiny_layer(seed=8, act=wl.BF16, wdt=wl.BF16, T=12)
    out, idx, w, _ = oracle.moe_forward(layer)
    perm = np.random.default_rng(1).permutation(layer.T)
    layer.x = layer.x[perm].copy()
    out_p, idx_p, w_p, _ = oracle.moe_forward(layer)
    assert np.array_equal(out_p, out[perm])
    assert np.array_equal(idx_p, idx[perm])
    assert np.array_equal(w_p, w[perm])


def test_linear_in_down_projection():
    layer = tiny_layer(seed=9)
    out, *_ = oracle.moe_forward(layer)
    layer.w_down = (layer.w_down * np.float32(2.0)).astype(np.float32)
    out2, *_ = oracle.moe_forward(layer)
    assert np.array_equal(out2, 2.0 * out)


def test_q8_0_equals_its_exact_dequantisation():
    """Q8_0 bytes and their fp32 dequantisation (exact: 11 x 8 bits) agree bit for bit."""
    layer = tiny_layer(seed=11, act=wl.BF16, wdt=wl.Q8_0, T=6, d=64, F=96)
    out_q, idx_q, w_q, _ = oracle.moe_forward(layer)
    for name in ("w_gate", "w_up", "w_down"):
        deq = decode(getattr(layer, name), wl.Q8_0)
        assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)
        setattr(layer, name, deq.astype(np.float32))
    layer.w_dtype = wl.F32
    out_f, idx_f, w_f, _ = oracle.moe_forward(layer)
    assert np.array_equal(idx_q, idx_f)
    assert np.array_equal(out_q, out_f)


def test_q8_0_fp16_scales_of_every_class_decode_exactly():
    """Block scales are IEEE binary16 (ggml's Q8_0, named in "zonos2.cpp
    internals", §Quantization: 32 int8 codes and one fp16 scale).  Scales set to subnormals (both
    signs, smallest and largest), the smallest normal, +-1 and zero must decode
    as numpy's float16 does: the layer on the Q8_0 bytes equals the layer on the
    fp32 values numpy decodes (each fp16 x int8 product is exact in fp32)."""
    layer = tiny_layer(seed=13, act=wl.BF16, wdt=wl.Q8_0, T=6, d=64, F=96)
    bits = np.array([0x0001, 0x0155, 0x03FF, 0x8200, 0x0400, 0x3C00, 0xBC00, 0x0000, 0x2E66],
                    np.uint16)
    for n, name in enumerate(("w_gate", "w_up", "w_down")):
        blocks = getattr(layer, name).copy()
        flat = blocks.reshape(-1, 34)
        pick = bits[(np.arange(flat.shape[0]) + n) % bits.size]
        flat[:, 0:2] = pick.view(np.uint8).reshape(-1, 2)
        setattr(layer, name, blocks)
    out_q, idx_q, _, _ = oracle.moe_forward(layer)
    assert np.abs(out_q).max() > 0
    for name in ("w_gate", "w_up", "w_down"):
        deq = decode(getattr(layer, name), wl.Q8_0)
        assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)
        setattr(layer, name, deq.astype(np.float32))
    layer.w_dtype = wl.F32
    out_f, idx_f, _, _ = oracle.moe_forward(layer)
    assert np.array_equal(idx_q, idx_f)
    assert np.array_equal(out_q, out_f)


def test_q8_0_block_encoding():
    w = np.zeros((2, 64), np.float32)
    w[0, :32] = np.linspace(-1, 1, 32)
    w[1, 32:] = 0.5
    blocks = wl.q8_0_quantize(w)
    assert blocks.shape == (2, 2, 34)
    deq = decode(blocks, wl.Q8_0)
    assert np.all(deq[0, 32:] == 0) and np.all(deq[1, :32] == 0)
    # scale = max|w|/127 stored in fp16; extreme values map to +-127
    s = np.float16(np.float32(1.0) / np.float32(127))
    assert blocks[0, 0, 2:].view(np.int8)[0] == -127
    np.testing.assert_allclose(deq[0, :32], w[0, :32], atol=float(s))


def test_permute_brute_force_and_invariants():
    rng = np.random.default_rng(12)
    for T, k, E in ((0, 2, 4), (1, 1, 1), (17, 2, 5), (100, 3, 9), (64, 4, 64)):
        idx = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)],
                       dtype=np.int32).reshape(T, k)
        counts, offsets, perm_tok, inv = oracle.permute(idx, E)
        assert counts.sum() == T * k
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        flat = idx.ravel()
        # brute force: stable sort of flat slots by expert
        order = sorted(range(T * k), key=lambda i: (flat[i], i))
        assert perm_tok.tolist() == [i // k for i in order]
        assert sorted(inv.tolist()) == list(range(T * k))
        for i in range(T * k):
            assert perm_tok[inv[i]] == i // k
            assert offsets[flat[i]] <= inv[i] < offsets[flat[i] + 1]


def test_margin_is_kth_minus_next_score():
    logits = np.array([[0.0, 3.0, 1.0, 2.0]])
    bias = np.array([0.5, 0, 0, 0], np.float32)
    idx, w, margin = oracle.selected_softmax(logits, bias, 2)
    assert idx[0].tolist() == [1, 3]
    assert margin[0] == 2.0 - 1.0


def test_invalid_arguments_raise():
    with pytest.raises(ValueError):
        oracle.selected_softmax(np.zeros((2, 4)), None, 5)
    with pytest.raises(ValueError):
        oracle.permute(np.array([[7]], np.int32), 4)


def test_multithreaded_equals_single_threaded():
    layer = tiny_layer(seed=13, act=wl.BF16, wdt=wl.BF16, T=33)
    a = oracle.moe_forward(layer, nthreads=1)
    b = oracle.moe_forward(layer, nthreads=7)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ---------------------------------------------- other scoring modes (next row f1)
# "New Community Model: ZONOS3-Mini (Zyphra) - #1271", §Framework change: the
# older modes apply a softmax or a sigmoid before ranking.  Reading (the pages
# give no formulas): p = softmax over all experts / sigmoid per expert, rank by
# p + bias, weigh by p of the selected experts, no renormalisation.

def _softmax_rows(l):
    from scipy.special import softmax
    return softmax(l, axis=1)


def _sigmoid(l):
    from scipy.special import expit
    return expit(l)


@pytest.mark.parametrize("k", [1, 2, 5])
def test_softmax_mode_weights_are_library_softmax_of_selected(k):
    rng = np.random.default_rng(40 + k)
    lg = rng.standard_normal((64, 12)) * 2.0
    b = (rng.standard_normal(12) * 0.05).astype(np.float32)
    idx, w, _ = oracle.route_scored(lg, b, k, oracle.SOFTMAX)
    p = _softmax_rows(lg)
    assert np.allclose(w, np.take_along_axis(p, idx, axis=1), rtol=0, atol=1e-15)
    # ranking: top-k of p + bias (library sort, ties to the lower index)
    s = p + b.astype(np.float64)
    ref = np.array([sorted(range(12), key=lambda e: (-s[t, e], e))[:k] for t in range(64)])
    assert np.array_equal(idx, ref)


@pytest.mark.parametrize("k", [1, 3])
def test_sigmoid_mode_weights_are_library_sigmoid(k):
    rng = np.random.default_rng(50 + k)
    lg = rng.standard_normal((64, 10)) * 3.0
    b = (rng.standard_normal(10) * 0.1).astype(np.float32)
    idx, w, _ = oracle.route_scored(lg, b, k, oracle.SIGMOID)
    sel = np.take_along_axis(lg, idx, axis=1)
    assert np.allclose(w, _sigmoid(sel), rtol=1e-15, atol=0)
    s = _sigmoid(lg) + b.astype(np.float64)
    ref = np.array([sorted(range(10), key=lambda e: (-s[t, e], e))[:k] for t in range(64)])
    assert np.array_equal(idx, ref)


def test_scoring_modes_zero_bias_same_set_as_selected_softmax():
    """Softmax and sigmoid are increasing, so with no bias every mode picks the
    same experts; softmax-mode weights are SelectedSoftmax's scaled by the
    selected experts' share of the full softmax."""
    rng = np.random.default_rng(60)
    lg = rng.standard_normal((100, 16))
    z = np.zeros(16, np.float32)
    i0, w0, _ = oracle.route_scored(lg, z, 3, oracle.SELECTED_SOFTMAX)
    i1, w1, _ = oracle.route_scored(lg, z, 3, oracle.SOFTMAX)
    i2, _, _ = oracle.route_scored(lg, z, 3, oracle.SIGMOID)
    assert np.array_equal(i0, i1) and np.array_equal(i0, i2)
    share = np.take_along_axis(_softmax_rows(lg), i0, axis=1).sum(axis=1, keepdims=True)
    assert np.allclose(w1, w0 * share, rtol=1e-13, atol=0)
    assert np.all(w1.sum(axis=1) < 1.0)   # not renormalised


def test_scoring_modes_rank_probabilities_plus_bias_worked_example():
    """Hand-derived: logits (0, 2, 3), bias (0.8, 0, 0), k = 1.  SelectedSoftmax
    ranks 0.8 < 2 < 3 and picks expert 2 (weight 1).  Softmax before rank:
    p = (1, e^2, e^3) / (1 + e^2 + e^3) = (0.03512, 0.25950, 0.70538), plus bias
    (0.83512, 0.25950, 0.70538): expert 0, weight 0.03512.  Sigmoid before rank:
    p = (0.5, 0.88080, 0.95257), plus bias (1.3, ...): expert 0, weight 1/2."""
    lg = np.array([[0.0, 2.0, 3.0]])
    b = np.array([0.8, 0.0, 0.0], np.float32)
    i0, w0, _ = oracle.route_scored(lg, b, 1, oracle.SELECTED_SOFTMAX)
    assert i0[0, 0] == 2 and w0[0, 0] == 1.0
    i1, w1, m1 = oracle.route_scored(lg, b, 1, oracle.SOFTMAX)
    assert i1[0, 0] == 0 and abs(w1[0, 0] - 0.0351190) < 1e-6
    assert abs(m1[0] - (0.8 + 0.0351190 - 0.7053845)) < 1e-6   # margin on p + bias
    i2, w2, _ = oracle.route_scored(lg, b, 1, oracle.SIGMOID)
    assert i2[0, 0] == 0 and w2[0, 0] == 0.5


def test_softmax_mode_k_equals_e_is_dense_softmax_and_bias_only_selects():
    rng = np.random.default_rng(70)
    lg = rng.standard_normal((20, 6))
    b = (rng.standard_normal(6) * 5).astype(np.float32)
    idx, w, margin = oracle.route_scored(lg, b, 6, oracle.SOFTMAX)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-15) and np.all(np.isinf(margin))
    # two different biases forcing the same set {1, 4}: identical weights
    f1 = np.array([0, 9, 0, 0, 8, 0], np.float32)
    f2 = np.array([0, 50, 0, 0, 40, 0], np.float32)
    for mode in (oracle.SOFTMAX, oracle.SIGMOID):
        ia, wa, _ = oracle.route_scored(lg, f1, 2, mode)
        ib, wb, _ = oracle.route_scored(lg, f2, 2, mode)
        assert np.array_equal(ia, ib) and np.all(ia == [1, 4]) and np.array_equal(wa, wb)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("k", [1, 2])
def test_scoring_modes_layer_matches_dense_brute_force(mode, k):
    layer = tiny_layer(seed=80 + k, k=k, bias_sd=0.2)
    out, idx, w, _ = oracle.moe_forward(layer, mode=mode)
    x = decode(layer.x, layer.act_dtype)
    wr = decode(layer.w_router, layer.act_dtype)
    lg = x @ wr.T
    p = _softmax_rows(lg) if mode == 1 else _sigmoid(lg)
    s = p + np.asarray(layer.bias, np.float64)
    wg = decode(layer.w_gate, layer.w_dtype)
    wu = decode(layer.w_up, layer.w_dtype)
    wd = decode(layer.w_down, layer.w_dtype)
    g = np.einsum("efi,ti->etf", wg, x)
    u = np.einsum("efi,ti->etf", wu, x)
    y = np.einsum("eif,etf->eti", wd, g / (1.0 + np.exp(-g)) * u)
    ref = np.zeros_like(x)
    for t in range(x.shape[0]):
        for e in sorted(range(layer.E), key=lambda e: (-s[t, e], e))[:k]:
            ref[t] += p[t, e] * y[e, t]
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


# ------------------------------------- dense SwiGLU layer (next row f2)
@pytest.mark.parametrize("act,wdt", [(wl.F32, wl.F32), (wl.BF16, wl.Q8_0)])
def test_one_expert_layer_is_the_dense_swiglu_ffn(act, wdt):
    """E = 1, k = 1: the weight is the softmax of one logit, exactly 1, so the
    layer is W_d (SiLU(W_g x) * (W_u x)) whatever the router holds."""
    layer = tiny_layer(seed=90, act=act, wdt=wdt, T=6, d=64, E=1, k=1, F=96)
    out, idx, w, _ = oracle.moe_forward(layer)
    assert np.all(idx == 0) and np.all(w == 1.0)
    x = decode(layer.x, act)
    wg = decode(layer.w_gate, wdt)[0]
    wu = decode(layer.w_up, wdt)[0]
    wd = decode(layer.w_down, wdt)[0]
    g, u = x @ wg.T, x @ wu.T
    ref = (g / (1.0 + np.exp(-g)) * u) @ wd.T
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())



# ------------------------------- affine 4-bit group-64 experts (next row f3)
def test_q4_a64_block_encoding_worked_example():
    """Hand-built group: w_i = (i mod 16) / 4 - 1 spans [-1, 2.75], so
    scale = 3.75 / 15 = 0.25 and bias = -1 (both exact in fp16), q_i = i mod 16
    exactly, byte j = q_2j | q_2j+1 << 4, and decoding gives w back exactly.
    A constant group has scale 0, bias = the value, codes 0."""
    w = np.array([(i % 16) / 4.0 - 1.0 for i in range(64)], np.float32)
    b = wl.q4_a64_quantize(w[None])[0, 0]
    assert b[0:2].view(np.float16)[0] == 0.25 and b[2:4].view(np.float16)[0] == -1.0
    assert np.array_equal(b[4:], np.array([(2 * j % 16) | ((2 * j + 1) % 16) << 4
                                           for j in range(32)], np.uint8))
    assert np.array_equal(decode(b[None, None], wl.Q4_A64)[0], w.astype(np.float64))
    c = wl.q4_a64_quantize(np.full((1, 64), 0.375, np.float32))[0, 0]
    assert c[0:2].view(np.float16)[0] == 0 and c[2:4].view(np.float16)[0] == 0.375
    assert not c[4:].any()


def test_q4_a64_error_within_half_a_step():
    rng = np.random.default_rng(91)
    w = rng.standard_normal((16, 256)).astype(np.float32)
    b = wl.q4_a64_quantize(w)
    deq = decode(b, wl.Q4_A64)
    step = np.repeat(b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64), 64, axis=-1)
    # half a step, plus the fp16 rounding of scale and bias (a few ulps of the range)
    assert np.all(np.abs(deq - w) <= 0.5 * step + 2e-3 * np.abs(w).max())


def test_q4_a64_layer_equals_its_exact_dequantisation():
    """The oracle on 4-bit bytes equals the oracle on fp32 weights holding the
    decoded values (exactly representable: fp16 scale x 4-bit code + fp16 bias)."""
    layer = tiny_layer(seed=92, act=wl.BF16, wdt=wl.Q4_A64, T=6, d=128, E=4, k=2, F=64)
    out_q, idx_q, _, _ = oracle.moe_forward(layer)
    import copy
    f = copy.copy(layer)
    f.w_dtype = wl.F32
    for n in ("w_gate", "w_up", "w_down"):
        v = decode(getattr(layer, n), wl.Q4_A64)
        assert np.array_equal(v.astype(np.float32).astype(np.float64), v)
        setattr(f, n, v.astype(np.float32))
    out_f, idx_f, _, _ = oracle.moe_forward(f)
    assert np.array_equal(idx_q, idx_f) and np.array_equal(out_q, out_f)


# ------------------------------------------- Q4_K super-blocks (next row f3)
def test_q4_k_super_block_worked_example():
    """A hand-built super-block: d = 0.5, dmin = 0.25, six-bit scales and mins
    chosen so that every bit of the 12 packed bytes is used (values >= 16 in
    sub-blocks 4-7 put bits in the top two bits of bytes 0-7), and code
    q = (i + 3j) mod 16 for value i of sub-block j.  The bytes are assembled
    here field by field from the format's description; value 32j + i must be
    0.5 * sc[j] * q - 0.25 * m[j], and the library's encoder helper must pack
    the same 12 bytes."""
    sc = [1, 2, 3, 63, 17, 33, 48, 5]
    mn = [0, 1, 62, 7, 16, 40, 3, 63]
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([0.5], np.float16).view(np.uint8)
    blk[2:4] = np.array([0.25], np.float16).view(np.uint8)
    for j in range(4):
        blk[4 + j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)     # sc[j]; top bits of sc[j+4]
        blk[8 + j] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)     # m[j];  top bits of m[j+4]
        blk[12 + j] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    q = np.array([[(i + 3 * j) % 16 for i in range(32)] for j in range(8)])
    for c in range(4):
        blk[16 + 32 * c:48 + 32 * c] = q[2 * c] | (q[2 * c + 1] << 4)
    assert np.array_equal(wl.q4_k_pack_scales(np.array(sc), np.array(mn)), blk[4:16])
    want = np.array([0.5 * sc[j] * q[j, i] - 0.25 * mn[j] for j in range(8) for i in range(32)])
    got = decode(blk[None, None], wl.Q4_K)[0]
    assert np.array_equal(got, want)
    # the oracle reads the same bytes: a one-expert layer with W_g = this row
    # against numpy on the hand values
    T, d, F = 3, 256, 256
    layer = tiny_layer(seed=93, act=wl.F32, wdt=wl.Q4_K, T=T, d=d, E=1, k=1, F=F)
    layer.w_gate = np.tile(blk, (1, F, 1)).reshape(1, F, 1, 144)
    x = decode(layer.x, wl.F32)
    g = x @ np.tile(want, (F, 1)).T
    u = x @ decode(layer.w_up, wl.Q4_K)[0].T
    ref = (g / (1.0 + np.exp(-g)) * u) @ decode(layer.w_down, wl.Q4_K)[0].T
    out, _, _, _ = oracle.moe_forward(layer)
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_q4_k_encoder_error_within_half_a_step():
    rng = np.random.default_rng(94)
    w = (rng.standard_normal((8, 512)) * 0.05).astype(np.float32)
    b = wl.q4_k_quantize(w)
    deq = decode(b, wl.Q4_K)
    d = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    # the largest step of each super-block: d * 63; half of it bounds the error
    # of values inside the sub-block's range, plus the six-bit rounding of the
    # scales and mins (one d / dmin unit each)
    dmin = b[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    bound = np.repeat(0.5 * 63 * d + 15 * d + dmin, 256, axis=-1)
    assert np.all(np.abs(deq - w) <= bound)
    assert np.sqrt(np.mean((deq - w) ** 2)) < 0.15 * np.sqrt(np.mean(w ** 2))



# ------------------------------------------- Q6_K super-blocks (next row f3)
def test_q6_k_super_block_worked_example():
    """A hand-built super-block: d = 0.25, scales[j] = 3j - 20 (negative and
    positive int8 scales), code q = (5v + 3) mod 64 for value v, so that every
    code and both top-bit positions occur.  The 210 bytes are assembled here
    value by value from the format's description (ql nibble, qh bit pair,
    scale byte, d); value v must be 0.25 * (3 (v // 16) - 20) * (q - 32), the
    library's packer must emit the same bytes, and the oracle reads them."""
    q = np.array([(5 * v + 3) % 64 for v in range(256)])
    scs = np.array([3 * j - 20 for j in range(16)])
    blk = np.zeros(210, np.uint8)
    for v in range(256):
        h, g, l = v // 128, (v % 128) // 32, v % 32
        lo, hi = q[v] & 15, q[v] >> 4
        blk[64 * h + l + 32 * (g % 2)] |= lo << (4 * (g // 2))
        blk[128 + 32 * h + l] |= hi << (2 * g)
    blk[192:208] = scs.astype(np.int8).view(np.uint8)
    blk[208:210] = np.array([0.25], np.float16).view(np.uint8)
    assert np.array_equal(wl.q6_k_pack(q.astype(np.uint8), scs.astype(np.int8), np.float16(0.25)), blk)
    want = np.array([0.25 * scs[v // 16] * (q[v] - 32) for v in range(256)])
    assert np.array_equal(decode(blk[None, None], wl.Q6_K)[0], want)
    T, d, F = 3, 256, 256
    layer = tiny_layer(seed=95, act=wl.F32, wdt=wl.Q6_K, T=T, d=d, E=1, k=1, F=F)
    layer.w_gate = np.tile(blk, (1, F, 1)).reshape(1, F, 1, 210)
    x = decode(layer.x, wl.F32)
    g = x @ np.tile(want, (F, 1)).T
    u = x @ decode(layer.w_up, wl.Q6_K)[0].T
    ref = (g / (1.0 + np.exp(-g)) * u) @ decode(layer.w_down, wl.Q6_K)[0].T
    out, _, _, _ = oracle.moe_forward(layer)
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_q6_k_encoder_error_within_half_a_step():
    rng = np.random.default_rng(96)
    w = (rng.standard_normal((8, 512)) * 0.05).astype(np.float32)
    b = wl.q6_k_quantize(w)
    deq = decode(b, wl.Q6_K)
    d = b[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
    sc = b[..., 192:208].copy().view(np.int8).astype(np.float64)
    # half a step of each 16-value group, plus the scale's rounding to a
    # multiple of d (at most d / 2 per unit of |q - 32| <= 32)
    bound = (0.5 * d[..., None] * np.abs(sc) + 16 * d[..., None]).repeat(16, axis=-1).reshape(8, 512)
    assert np.all(np.abs(deq - w) <= bound)
    assert np.sqrt(np.mean((deq - w) ** 2)) < 0.03 * np.sqrt(np.mean(w ** 2))


# ------------------------------------------- fp8 (E4M3) experts (next row f3)
# code -> value, written from the E4M3 definition (sign, 4 exponent bits with
# bias 7, 3 mantissa bits, exponent field 0 subnormal, no infinities)
E4M3_WORKED = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
               0x30: 0.5, 0x38: 1.0, 0x3C: 1.5, 0x3F: 1.875, 0x40: 2.0, 0x57: 15.0, 0x7E: 448.0,
               0x80: -0.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xC4: -3.0, 0xFE: -448.0}


def test_fp8_e4m3_worked_codes_and_library_decode():
    """Hand-derived E4M3 values agree with torch's float8_e4m3fn (the tests'
    decoder), which then decodes every finite code."""
    import torch
    codes = np.array(sorted(E4M3_WORKED), np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert lib.tolist() == [E4M3_WORKED[c] for c in codes.tolist()]
    allc = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.isnan(allc[[0x7F, 0xFF]]).all() and np.isfinite(np.delete(allc, [0x7F, 0xFF])).all()
    assert np.abs(allc[np.isfinite(allc)]).max() == 448.0


def test_fp8_every_code_through_a_layer():
    """One expert whose W_g rows hold every finite E4M3 code (NaN codes
    replaced by zero) under scales of both signs' magnitudes: the oracle's
    layer output against a numpy forward on the torch-decoded weights."""
    T, d, F = 4, 256, 64
    layer = tiny_layer(seed=97, act=wl.F32, wdt=wl.FP8, T=T, d=d, E=1, k=1, F=F)
    rows = np.zeros((1, F, 4 + d), np.uint8)
    codes = np.arange(256, dtype=np.uint8)
    codes[[0x7F, 0xFF]] = 0
    for f in range(F):
        rows[0, f, 4:] = np.roll(codes, 5 * f)
        rows[0, f, 0:4] = np.array([2.0 ** -(f % 7) * (1 + f / 64.0)], np.float32).view(np.uint8)
    layer.w_gate = rows
    x = decode(layer.x, wl.F32)
    g = x @ decode(layer.w_gate, wl.FP8)[0].T
    u = x @ decode(layer.w_up, wl.FP8)[0].T
    ref = (g / (1.0 + np.exp(-g)) * u) @ decode(layer.w_down, wl.FP8)[0].T
    out, _, _, _ = oracle.moe_forward(layer)
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_fp8_encoder_error_within_half_a_step():
    rng = np.random.default_rng(98)
    w = (rng.standard_normal((8, 512)) * 0.05).astype(np.float32)
    w[3] = 0.0
    b = wl.fp8_quantize(w)
    deq = decode(b, wl.FP8)
    s = b[..., 0:4].copy().view(np.float32)[..., 0].astype(np.float64)
    assert s[3] == 1.0 and np.all(deq[3] == 0.0)
    v = np.abs(w / s[:, None].astype(np.float32)).astype(np.float64)
    # half the E4M3 spacing at |v|: 2^(floor(log2 v) - 4) for normals, 2^-10 below 2^-6
    half = np.where(v >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 4), 2.0 ** -10)
    assert np.all(np.abs(deq - w) <= half * s[:, None] * (1 + 1e-6))
    # each nonzero row's largest magnitude lands on 448 (to within the scale's rounding)
    for r in range(8):
        if r != 3:
            assert abs(np.abs(deq[r]).max() / s[r] - 448.0) <= 448.0 * 2.0 ** -4
