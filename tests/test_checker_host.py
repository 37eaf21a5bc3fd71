"""The GPU parity checks must reject wrong results (CPU, no GPU).

tests/helpers.py holds the checks every GPU parity test uses: routing indices
exact beyond the ranking margin, weights within 2e-6, and the output within
TOL * RMS of the oracle, with near-tie tokens re-evaluated on the experts the
GPU chose.  Here the "GPU result" is the oracle's own, with a mistake planted:
each planted mistake must fail the check, and the unchanged result must pass.
"""
import numpy as np
import pytest

import oracle
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
from helpers import MARGIN, TOL, check_output, compare_routing


def _layer(seed=5, T=12, E=8, k=2):
    return wl.make_custom_layer(seed, T, 64, E, k, 96, wl.F32, wl.F32, bias_sd=0.3)


def _with_near_tie(layer, t=0):
    """Move the (k+1)-th expert of token t to within 1e-4 of the k-th score."""
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    score = logits[t] + layer.bias.astype(np.float64)
    order = sorted(range(layer.E), key=lambda e: (-score[e], e))
    kth, nxt = order[layer.k - 1], order[layer.k]
    layer.bias = layer.bias.copy()
    layer.bias[nxt] = np.float32(score[kth] - 1e-4 - logits[t, nxt])
    return kth, nxt


def test_unchanged_result_passes():
    layer = _layer()
    out, idx, w, margin = oracle.moe_forward(layer)
    compare_routing(idx, w.astype(np.float32), idx, w, margin, layer.k)
    check_output(out.astype(np.float32), layer, out, idx, margin, idx_gpu=idx)


def test_output_error_beyond_tolerance_fails():
    layer = _layer()
    out, idx, w, margin = oracle.moe_forward(layer)
    bad = out.copy()
    rms = np.sqrt(np.mean(out ** 2))
    bad[3, 7] += 2 * TOL[wl.F32] * rms
    with pytest.raises(AssertionError, match="max\\|err\\|"):
        check_output(bad, layer, out, idx, margin, idx_gpu=idx)


def test_unweighted_combine_fails():
    """Every expert output added with weight 1 instead of its routing weight."""
    layer = _layer()
    out, idx, w, margin = oracle.moe_forward(layer)
    bad = oracle.expert_combine(layer.x, layer.act_dtype, idx, np.ones_like(w), layer.w_gate,
                                layer.w_up, layer.w_down, layer.w_dtype, layer.E, layer.F)
    with pytest.raises(AssertionError):
        check_output(bad, layer, out, idx, margin, idx_gpu=idx)


def test_other_expert_on_a_safe_margin_token_fails():
    layer = _layer()
    out, idx, w, margin = oracle.moe_forward(layer)
    t = int(np.argmax(margin))
    assert margin[t] >= MARGIN
    idx_bad = idx.copy()
    idx_bad[t, -1] = next(e for e in range(layer.E) if e not in idx[t])
    with pytest.raises(AssertionError, match="routed differently"):
        compare_routing(idx_bad, w.astype(np.float32), idx, w, margin, layer.k)
    with pytest.raises(AssertionError, match="safe-margin"):
        check_output(out, layer, out, idx, margin, idx_gpu=idx_bad)


def test_routing_weight_off_or_slots_swapped_fails():
    layer = _layer()
    out, idx, w, margin = oracle.moe_forward(layer)
    t = int(np.argmax(margin))
    w_bad = w.astype(np.float32).copy()
    w_bad[t, 0] += 1e-5
    with pytest.raises(AssertionError):
        compare_routing(idx, w_bad, idx, w, margin, layer.k)
    idx_swapped = idx.copy()
    idx_swapped[t] = idx[t, ::-1]
    with pytest.raises(AssertionError):
        compare_routing(idx_swapped, w.astype(np.float32), idx, w, margin, layer.k)


def test_k1_weight_not_one_fails():
    layer = _layer(k=1)
    out, idx, w, margin = oracle.moe_forward(layer)
    w_bad = w.astype(np.float32).copy()
    w_bad[np.argmin(margin), 0] = np.nextafter(np.float32(1), np.float32(0))
    with pytest.raises(AssertionError):
        compare_routing(idx, w_bad, idx, w, np.full_like(margin, -1.0), 1)


def test_near_tie_accepts_either_set_but_only_with_its_own_output():
    layer = _layer(seed=6)
    kth, nxt = _with_near_tie(layer, t=0)
    out, idx, w, margin = oracle.moe_forward(layer)
    assert margin[0] < MARGIN and idx[0, -1] == kth
    # the GPU may pick the runner-up: the check re-runs the oracle on its set
    idx_alt = idx.copy()
    idx_alt[0, -1] = nxt
    logits = oracle.router_logits(layer.x[:1], layer.act_dtype, layer.w_router, layer.E)
    w_alt = oracle.softmax_of_set(logits, idx_alt[:1])
    out_alt = out.copy()
    out_alt[0] = oracle.expert_combine(layer.x[:1], layer.act_dtype, idx_alt[:1], w_alt,
                                       layer.w_gate, layer.w_up, layer.w_down, layer.w_dtype,
                                       layer.E, layer.F)[0]
    compare_routing(idx_alt, w.astype(np.float32), idx, w, margin, layer.k)
    check_output(out_alt, layer, out, idx, margin, idx_gpu=idx_alt)
    # ... but claiming the runner-up while returning the original set's output fails
    with pytest.raises(AssertionError, match="max\\|err\\|"):
        check_output(out, layer, out, idx, margin, idx_gpu=idx_alt)


def _near_tie_case(seed=6, k=2, E=8):
    layer = _layer(seed=seed, k=k, E=E)
    kth, nxt = _with_near_tie(layer, t=0)
    out, idx, w, margin = oracle.moe_forward(layer)
    logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    return layer, out, idx, w, margin, logits, kth, nxt


def test_near_tie_swap_outside_the_tie_band_fails():
    """A near-tie token may trade its k-th expert for the runner-up, not for an
    expert that scores well below the tie."""
    layer, out, idx, w, margin, logits, kth, nxt = _near_tie_case()
    score = logits[0] + layer.bias.astype(np.float64)
    s_k = score[kth]
    far = [e for e in range(layer.E) if e not in idx[0] and score[e] < s_k - 10 * MARGIN]
    assert far
    idx_bad = idx.copy()
    idx_bad[0, -1] = far[0]
    w_bad = w.astype(np.float32).copy()
    w_bad[:1] = oracle.softmax_of_set(logits[:1], idx_bad[:1])
    with pytest.raises(AssertionError, match="below the tie band"):
        compare_routing(idx_bad, w_bad, idx, w, margin, layer.k, logits=logits, bias=layer.bias)
    out_bad = out.copy()
    out_bad[0] = oracle.expert_combine(layer.x[:1], layer.act_dtype, idx_bad[:1], w_bad[:1],
                                       layer.w_gate, layer.w_up, layer.w_down, layer.w_dtype,
                                       layer.E, layer.F)[0]
    with pytest.raises(AssertionError, match="below the tie band"):
        check_output(out_bad, layer, out, idx, margin, idx_gpu=idx_bad)


def test_near_tie_dropping_an_expert_above_the_band_fails():
    """Swapping out the top expert (well above the tie) for the runner-up fails."""
    layer, out, idx, w, margin, logits, kth, nxt = _near_tie_case(k=2)
    idx_bad = idx.copy()
    idx_bad[0, 0] = nxt            # drops the first-ranked expert, keeps the k-th
    w_bad = w.astype(np.float32).copy()
    w_bad[:1] = oracle.softmax_of_set(logits[:1], idx_bad[:1])
    with pytest.raises(AssertionError, match="above the tie band dropped"):
        compare_routing(idx_bad, w_bad, idx, w, margin, layer.k, logits=logits, bias=layer.bias)


def test_near_tie_set_with_wrong_weights_fails():
    """The runner-up set is valid, but only with its own softmax weights."""
    layer, out, idx, w, margin, logits, kth, nxt = _near_tie_case()
    idx_alt = idx.copy()
    idx_alt[0, -1] = nxt
    w_alt = w.astype(np.float32).copy()
    w_alt[:1] = oracle.softmax_of_set(logits[:1], idx_alt[:1])
    compare_routing(idx_alt, w_alt, idx, w, margin, layer.k, logits=logits, bias=layer.bias)
    # the original set's weights on the runner-up set are wrong (the logits differ by far more
    # than 2e-6)
    with pytest.raises(AssertionError):
        compare_routing(idx_alt, w.astype(np.float32), idx, w, margin, layer.k, logits=logits,
                        bias=layer.bias)


def test_near_tie_repeated_expert_fails():
    layer, out, idx, w, margin, logits, kth, nxt = _near_tie_case(k=3, E=8)
    idx_bad = idx.copy()
    idx_bad[0, -1] = idx_bad[0, 0]
    with pytest.raises(AssertionError, match="repeated expert"):
        compare_routing(idx_bad, w.astype(np.float32), idx, w, margin, layer.k, logits=logits,
                        bias=layer.bias)
