"""Shared test utilities: device upload of workload arrays and parity checks."""
import numpy as np

from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

# Output tolerances: max|gpu - oracle| <= TOL * RMS(oracle output).
TOL = {wl.F32: 1e-4, wl.BF16: 2e-2, wl.Q8_0: 2e-2, wl.Q4_A64: 2e-2}
# Routing indices must match exactly where the oracle's k-th vs (k+1)-th
# ranking-score margin is at least this.
MARGIN = 1e-3


def to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def upload_layer(layer, dev):
    """Device tensors for moe_forward; Q8_0 weights are packed on the device."""
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    t = dict(x=to_dev(layer.x, dev), w_router=to_dev(layer.w_router, dev),
             bias=to_dev(layer.bias, dev))
    if layer.w_dtype in (wl.Q8_0, wl.Q4_A64):
        E, F, d = layer.E, layer.F, layer.d
        pack = pkg.moe_pack_q8_0 if layer.w_dtype == wl.Q8_0 else pkg.moe_pack_q4_a64
        t["w_gate"] = pack(to_dev(layer.w_gate.reshape(-1), dev), E * F, d)
        t["w_up"] = pack(to_dev(layer.w_up.reshape(-1), dev), E * F, d)
        t["w_down"] = pack(to_dev(layer.w_down.reshape(-1), dev), E * d, F)
    else:
        for n in ("w_gate", "w_up", "w_down"):
            t[n] = to_dev(getattr(layer, n), dev)
    return t


def gpu_forward(layer, dev, path=0, t=None, out=None, workspace=None, scoring=0):
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    t = upload_layer(layer, dev) if t is None else t
    return pkg.moe_forward(t["x"], t["w_router"], t["bias"], t["w_gate"], t["w_up"], t["w_down"],
                           layer.k, F=layer.F, w_dtype=layer.w_dtype, path=path, out=out,
                           workspace=workspace, scoring=scoring)


def weights_of_set(logits, idx, mode=0):
    """Weights the scoring mode gives a fixed selected set (fp64): softmax of
    the set's logits (0), the full softmax at the set (1), sigmoid (2)."""
    import oracle
    if mode == 0:
        return oracle.softmax_of_set(logits, idx)
    if mode == 1:
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        return np.take_along_axis(z / z.sum(axis=1, keepdims=True), idx, axis=1)
    return 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx, axis=1)))


def sub_layer(layer, rows):
    """The same layer restricted to token rows `rows` (oracle sampling)."""
    import copy
    s = copy.copy(layer)
    s.x = np.ascontiguousarray(layer.x[rows])
    s.T = len(rows)
    return s


def compare_routing(idx_gpu, w_gpu, idx_ref, w_ref, margin, k, mode=0):
    """Indices exact where the margin is safe; weights close there."""
    ok = margin >= MARGIN
    assert np.array_equal(idx_gpu[ok], idx_ref[ok]), \
        f"{int((idx_gpu[ok] != idx_ref[ok]).any(1).sum())} tokens routed differently"
    np.testing.assert_allclose(w_gpu[ok], w_ref[ok], rtol=0, atol=2e-6)
    if k == 1 and mode == 0:
        assert np.all(w_gpu == 1.0)
    return ok


def check_output(out_gpu, layer, ref, idx_ref, margin, idx_gpu=None, rows=None, mode=0):
    """max|gpu - oracle| <= TOL * RMS(oracle), re-evaluating near-tie tokens.

    A token whose ranking margin is below MARGIN may legitimately select a
    different expert set on the GPU (fp32 vs fp64 scores); for those the oracle
    is re-run with the GPU's selected set.
    """
    import oracle
    ref = ref.copy()
    if idx_gpu is not None:
        diff = np.where((idx_gpu != idx_ref).any(1))[0]
        if len(diff):
            assert np.all(margin[diff] < MARGIN), "routing differs on a safe-margin token"
            sub = sub_layer(layer, diff)
            logits = oracle.router_logits(sub.x, layer.act_dtype, layer.w_router, layer.E)
            w = weights_of_set(logits, idx_gpu[diff], mode)
            ref[diff] = oracle.expert_combine(sub.x, layer.act_dtype, idx_gpu[diff], w,
                                              layer.w_gate, layer.w_up, layer.w_down,
                                              layer.w_dtype, layer.E, layer.F)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(out_gpu.astype(np.float64) - ref)
    tol = TOL[layer.w_dtype if layer.act_dtype != wl.F32 else wl.F32]
    assert err.max() <= tol * rms, f"max|err| {err.max():.3e} > {tol} * RMS {rms:.3e}"
    return err.max() / rms
