"""Fit the selection bias of the full-size ZONOS3-Mini prefill layers so that
their expert loads follow Zipf(s = 1.1) over the 64 expert ranks, and write
the fixture zipf_bias_zonos3_mini_prefill.txt beside this script.

Inputs of record: layer i's x and W_r from workloads.zipf_host_inputs (host
seeds), rank r held by expert order[r].  Target: the top-2 assignments of
the T = 8192 tokens split as T*k * r^-1.1 / sum_r r^-1.1.  Procedure (fixed,
deterministic): the router logits in fp64 from the bf16 inputs, once
(oracle.router_logits); b_e = log p_rank(e); then 200 rounds of
    b_e <- b_e + 0.5 * (log target_e - log max(count_e, 0.5)),
each count taken from SelectedSoftmax routing with the current bias rounded
to fp32, the bias the layer is given (oracle.selected_softmax: rank by
logit + bias, keep the top 2).  The bias after the last round, as fp32, and
the counts it achieves are the workload of record.

Routing here is the oracle's only; the counting and the update are plain
numpy.  Run:  python tests/golden/fit_zipf_bias.py   (a few seconds)
"""
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl  # noqa: E402

FIXTURE = os.path.join(HERE, "zipf_bias_zonos3_mini_prefill.txt")
ROUNDS = 200
STEP = 0.5


def layer_logits(w, layer):
    x, wr, order = wl.zipf_host_inputs(w, layer)
    logits = oracle.router_logits(wl.f32_to_bf16_bits(x), wl.BF16, wl.f32_to_bf16_bits(wr), w.E)
    return logits, order


def counts_of(logits, bias, E, k):
    idx, _, _ = oracle.selected_softmax(logits, np.asarray(bias, dtype=np.float32), k)
    return np.bincount(idx.reshape(-1), minlength=E)


def fit(logits, order, E, T, k):
    target = np.empty(E)
    target[order] = wl.zipf_targets(E, T, k)          # expert order[r] holds rank r + 1
    b = np.log(target / (T * k))
    for _ in range(ROUNDS):
        cnt = counts_of(logits, b.astype(np.float32), E, k)
        b = b + STEP * (np.log(target) - np.log(np.maximum(cnt, 0.5)))
    b32 = b.astype(np.float32)
    return b32, counts_of(logits, b32, E, k), target


def main():
    w = wl.WORKLOADS["zonos3_mini_prefill"]
    lines = ["# Selection bias of the full-size ZONOS3-Mini prefill layers (T=8192, d=1024,",
             "# E=64, k=2), fitted with the oracle's SelectedSoftmax routing so that the",
             "# expert loads follow Zipf(s=1.1) over the 64 ranks; written by",
             "# tests/golden/fit_zipf_bias.py (see its docstring for the procedure).",
             "# Per layer: 'bias <i>' then 64 fp32 values (expert order), 'counts <i>' then",
             "# the 64 achieved assignment counts, 'target <i>' the Zipf targets."]
    for layer in range(w.layers):
        logits, order = layer_logits(w, layer)
        b, cnt, target = fit(logits, order, w.E, w.T, w.k)
        lines.append(f"bias {layer} " + " ".join(repr(float(v)) for v in b))
        lines.append(f"counts {layer} " + " ".join(str(int(v)) for v in cnt))
        lines.append(f"target {layer} " + " ".join(f"{v:.3f}" for v in target))
        rel = np.abs(cnt - target) / target
        print(f"layer {layer}: top {cnt.max()} (target {target.max():.0f}), bottom {cnt.min()} "
              f"(target {target.min():.1f}), max |count/target - 1| {rel.max():.3f}")
    with open(FIXTURE, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", FIXTURE)


def load(path=FIXTURE):
    """{layer: (bias fp32 [E], counts [E], target [E])} from the fixture."""
    out = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        key, layer, *vals = line.split()
        rec = out.setdefault(int(layer), {})
        rec[key] = np.array([float(v) for v in vals])
    return {i: (r["bias"].astype(np.float32), r["counts"].astype(np.int64), r["target"])
            for i, r in out.items()}


if __name__ == "__main__":
    main()
