"""The fitted selection bias of the full-size ZONOS3-Mini prefill layers
(tests/golden/zipf_bias_zonos3_mini_prefill.txt): its recorded loads are
what the oracle's SelectedSoftmax routing gives on the layers' inputs, and
they follow the Zipf(s = 1.1) targets over the 64 expert ranks."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import fit_zipf_bias as fz  # noqa: E402
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl  # noqa: E402

W = wl.WORKLOADS["zonos3_mini_prefill"]


def test_fixture_covers_every_layer_with_the_zipf_targets():
    rec = fz.load()
    assert sorted(rec) == list(range(W.layers))
    for layer, (b, cnt, target) in rec.items():
        _, _, order = wl.zipf_host_inputs(W, layer)
        want = np.empty(W.E)
        want[order] = wl.zipf_targets(W.E, W.T, W.k)
        assert np.allclose(target, want, atol=1e-3)
        assert b.shape == (W.E,) and np.all(np.isfinite(b))
        assert cnt.sum() == W.T * W.k
        # every expert is used; the loads follow the targets: 1.5 % of the
        # assignments off target in total, the 8 busiest ranks within 2.5 %
        assert cnt.min() > 0
        assert np.abs(cnt - target).sum() / cnt.sum() < 0.02
        top = np.argsort(-target)[:8]
        assert np.all(np.abs(cnt[top] / target[top] - 1.0) < 0.025)


def test_recorded_loads_are_the_oracles_routing_of_layer_0():
    rec = fz.load()
    b, cnt, _ = rec[0]
    logits, _ = fz.layer_logits(W, 0)
    assert np.array_equal(fz.counts_of(logits, b, W.E, W.k), cnt)
