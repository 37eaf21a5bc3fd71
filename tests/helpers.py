"""Shared test utilities: device upload of workload arrays and parity checks."""
import numpy as np

from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

# Output tolerances: max|gpu - oracle| <= TOL * RMS(oracle output).
TOL = {wl.F32: 1e-4, wl.BF16: 2e-2, wl.Q8_0: 2e-2, wl.Q4_A64: 2e-2, wl.Q4_K: 2e-2, wl.Q6_K: 2e-2,
       wl.FP8: 2e-2}
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
    if layer.w_dtype in (wl.Q8_0, wl.Q4_A64, wl.Q4_K, wl.Q6_K, wl.FP8):
        E, F, d = layer.E, layer.F, layer.d
        pack = {wl.Q8_0: pkg.moe_pack_q8_0, wl.Q4_A64: pkg.moe_pack_q4_a64,
                wl.Q4_K: pkg.moe_pack_q4_k, wl.Q6_K: pkg.moe_pack_q6_k,
                wl.FP8: pkg.moe_pack_fp8}[layer.w_dtype]
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


def ranking_scores(logits, bias, mode=0):
    """The oracle's fp64 ranking scores of a scoring mode: logit + bias (0),
    softmax over all experts + bias (1), sigmoid + bias (2)."""
    b = 0.0 if bias is None else np.asarray(bias, np.float64)[None, :]
    if mode == 0:
        return logits + b
    if mode == 1:
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True) + b
    return 1.0 / (1.0 + np.exp(-logits)) + b


def assert_near_tie_sets_valid(scores, idx_gpu, idx_ref, margin, k):
    """Tokens whose GPU set differs from the oracle's: the oracle margin must be
    below MARGIN, and the GPU set must be a correct resolution of the tie --
    k distinct experts, every expert scoring above s_k + MARGIN kept, and every
    kept expert scoring at least s_k - MARGIN (s_k: the oracle's k-th highest
    score of that token)."""
    diff = np.where((idx_gpu != idx_ref).any(1))[0]
    if not len(diff):
        return diff
    assert np.all(margin[diff] < MARGIN), "routing differs on a safe-margin token"
    for t in diff:
        sel = [int(e) for e in idx_gpu[t]]
        assert len(set(sel)) == k, f"token {t}: repeated expert in {sel}"
        assert all(0 <= e < scores.shape[1] for e in sel), f"token {t}: expert out of range"
        s_k = scores[t, idx_ref[t, k - 1]]
        must = np.where(scores[t] > s_k + MARGIN)[0]
        assert set(must.tolist()) <= set(sel), \
            f"token {t}: experts {sorted(set(must.tolist()) - set(sel))} above the tie band dropped"
        low = [e for e in sel if scores[t, e] < s_k - MARGIN]
        assert not low, f"token {t}: experts {low} below the tie band kept"
    return diff


def compare_routing(idx_gpu, w_gpu, idx_ref, w_ref, margin, k, mode=0, logits=None, bias=None,
                    w_atol=2e-6):
    """Indices exact where the margin is safe; weights close there (w_atol).
    With the oracle's logits (and the bias), tokens under the margin whose set
    differs are checked too: a valid resolution of the tie, weighted as the
    scoring mode weighs that set."""
    ok = margin >= MARGIN
    assert np.array_equal(idx_gpu[ok], idx_ref[ok]), \
        f"{int((idx_gpu[ok] != idx_ref[ok]).any(1).sum())} tokens routed differently"
    np.testing.assert_allclose(w_gpu[ok], w_ref[ok], rtol=0, atol=w_atol)
    if k == 1 and mode == 0:
        assert np.all(w_gpu == 1.0)
    if logits is not None:
        scores = ranking_scores(logits, bias, mode)
        diff = assert_near_tie_sets_valid(scores, idx_gpu, idx_ref, margin, k)
        if len(diff):
            w_set = weights_of_set(logits[diff], idx_gpu[diff], mode)
            np.testing.assert_allclose(w_gpu[diff], w_set, rtol=0, atol=w_atol)
        same = ~ok & ~(idx_gpu != idx_ref).any(1)
        np.testing.assert_allclose(w_gpu[same], w_ref[same], rtol=0, atol=w_atol)
    return ok


def check_output(out_gpu, layer, ref, idx_ref, margin, idx_gpu=None, rows=None, mode=0):
    """max|gpu - oracle| <= TOL * RMS(oracle), re-evaluating near-tie tokens.

    A token whose ranking margin is below MARGIN may legitimately select a
    different expert set on the GPU (fp32 vs fp64 scores).  For those the GPU's
    set must be a valid resolution of the tie (assert_near_tie_sets_valid), and
    the oracle is re-run with that set.  idx_gpu should be the indices the
    layer itself used (read back from its workspace).
    """
    import oracle
    ref = ref.copy()
    if idx_gpu is not None:
        diff = np.where((idx_gpu != idx_ref).any(1))[0]
        if len(diff):
            assert np.all(margin[diff] < MARGIN), "routing differs on a safe-margin token"
            sub = sub_layer(layer, diff)
            logits = oracle.router_logits(sub.x, layer.act_dtype, layer.w_router, layer.E)
            scores = ranking_scores(logits, layer.bias, mode)
            assert_near_tie_sets_valid(scores, idx_gpu[diff], idx_ref[diff], margin[diff],
                                       idx_ref.shape[1])
            w = weights_of_set(logits, idx_gpu[diff], mode)
            ref[diff] = oracle.expert_combine(sub.x, layer.act_dtype, idx_gpu[diff], w,
                                              layer.w_gate, layer.w_up, layer.w_down,
                                              layer.w_dtype, layer.E, layer.F)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(out_gpu.astype(np.float64) - ref)
    tol = TOL[layer.w_dtype if layer.act_dtype != wl.F32 else wl.F32]
    assert err.max() <= tol * rms, f"max|err| {err.max():.3e} > {tol} * RMS {rms:.3e}"
    return err.max() / rms


def gpu_forward_views(layer, dev, path=0, t=None, scoring=0, out=None):
    """moe_forward with a workspace of its own, then the routing and grouping
    that call's kernels left in the workspace (moe_workspace_views), as numpy
    arrays: (out, {topk_idx, topk_w, counts, offsets, perm_tok, inv, perm_w})."""
    import torch
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    t = upload_layer(layer, dev) if t is None else t
    args = (layer.T, layer.d, layer.E, layer.k, layer.F, layer.act_dtype, layer.w_dtype)
    ws = torch.empty(max(pkg.moe_workspace_size(*args), 256), dtype=torch.uint8, device=dev)
    o = gpu_forward(layer, dev, path=path, t=t, out=out, workspace=ws, scoring=scoring)
    torch.cuda.synchronize()
    assert pkg.moe_check(ws) == 0
    r = pkg.read_routing(ws, *args)
    return o.cpu().numpy(), {n: v.cpu().numpy() for n, v in r.items()}


def check_routing_views(r, layer, mode=0, logits=None, w_atol=2e-6):
    """The routing and grouping a layer call wrote, against the oracle:
    indices exact beyond the margin (near ties: a valid resolution), weights
    within 2e-6, counts / offsets / perm_tok / inv bit-exact against the
    oracle's grouping of the call's own indices, and perm_w bit-equal to the
    call's routing weight of each grouped row's slot.  Returns the oracle's
    (idx, w, margin)."""
    import oracle
    if logits is None:
        logits = oracle.router_logits(layer.x, layer.act_dtype, layer.w_router, layer.E)
    idx_ref, w_ref, margin = oracle.route_scored(logits, layer.bias, layer.k, mode)
    idx = r["topk_idx"]
    compare_routing(idx, r["topk_w"], idx_ref, w_ref, margin, layer.k, mode, logits=logits,
                    bias=layer.bias, w_atol=w_atol)
    c, o, p, i = oracle.permute(idx, layer.E)
    assert np.array_equal(r["counts"], c), "counts differ from the grouping of the call's routing"
    assert np.array_equal(r["offsets"], o), "offsets differ"
    assert np.array_equal(r["perm_tok"], p), "perm_tok differs"
    assert np.array_equal(r["inv"], i), "inv differs"
    slot_of_row = np.argsort(i, kind="stable")
    assert np.array_equal(r["perm_w"], r["topk_w"].reshape(-1)[slot_of_row]), "perm_w differs"
    return idx_ref, w_ref, margin
