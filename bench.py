"""Benchmark of the GB300 MoE FFN layer with SelectedSoftmax routing.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--T T] [--no-graph]

A step is one pass of the whole layer (routing, grouping, expert FFN,
combine) over every layer of the workload's stack, on synthetic inputs
resident in HBM.  The default workload is the ZONOS3-Mini-shaped decode step:
T=128 rows, d=1024, E=64, top-2, F=512, bf16, 10 independent MoE layers
back to back (2.0 GB of expert weights per step, far above the 129 MB L2, so
every step reads its weights from HBM).  value = layer-tokens per second
(T x layers x steps / time).  One JSON line is printed by rank 0.

With the default workload the line also carries a "workloads" list: every
other configuration (tiny fp32; ZONOS2-shaped decode at T = 1, 8 and 64; the
ZONOS3-Mini-shaped prefill; the ZONOS2-shaped Q8_0 prefill), each measured
alone on rank 0's GPU -- µs per layer, tokens/s, the layer's roofline
fraction, the dominant kernel's fraction -- with the oracle's tokens/s on the
host cores beside it (median of 3 passes over a token sample).

--impl reference times the CPU fp64 oracle (the only reference this library
has) on the machine's host cores, on bounded token samples of the same workload.
Under torchrun each rank runs an independent replica (no collective on the
data path); timing is max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode HBM GB/s and prefill TFLOPS as % of GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="zonos3_mini_decode")
    p.add_argument("--T", type=int, default=None)
    p.add_argument("--layers", type=int, default=None)
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--side", default=None, help=argparse.SUPPRESS)   # NAME[:T], one side config
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the per-configuration block (the other workloads, measured alone)")
    p.add_argument("--dense", action="store_true",
                   help="a dense SwiGLU layer of the workload's d and F (one expert, k = 1) "
                        "through moe_ffn_dense")
    p.add_argument("--scoring", default="selected_softmax",
                   choices=["selected_softmax", "softmax", "sigmoid"],
                   help="router scoring mode (SelectedSoftmax, or softmax / sigmoid before rank)")
    return p.parse_args()


def max_over_ranks(t_ms, world, device):
    """The slowest rank's time: the whole job ends when it does (world > 1:
    an all-reduce over the initialised process group)."""
    if world <= 1:
        return float(t_ms)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(t_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(tokens_per_step_per_rank, world, ms_per_step):
    """Whole-job tokens/s: every rank processes its own tokens each step."""
    return tokens_per_step_per_rank * world / (ms_per_step * 1e-3)


def layer_roofline_frac(bytes_, flops, seconds, hbm_gbs, tflops):
    """Achieved fraction of the layer's roofline: the slower of its bytes at HBM
    bandwidth and its flops at the tensor peak, over the measured time."""
    bound = max(bytes_ / (hbm_gbs * 1e9), flops / (tflops * 1e12))
    return bound / seconds


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, key):
    for k, v in peaks.items():
        if k == key and isinstance(v, (int, float)):
            return float(v)
    # tolerate nested layouts {"hbm_gbs": {"value": ..}}
    v = peaks.get(key)
    if isinstance(v, dict) and "value" in v:
        return float(v["value"])
    return FALLBACK_PEAKS[key]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- algorithmic
def algorithmic(w, T, counts_per_layer):
    """Algorithmic bytes/flops per stage for one step (sum over the stack).

    Bytes: each active expert's weights once, x, W_r, bias, fp32 output.
    Flops: 2*T*d*E (router) + 2*T*k*3*d*F (experts).
    """
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    asz = wl.act_bytes(w.act_dtype)
    per_w = wl.weight_bytes_per_expert(w.d, w.F, w.w_dtype)
    gu_w, dn_w = per_w * 2 // 3, per_w // 3
    x_b, wr_b, out_b, b_b = T * w.d * asz, w.E * w.d * asz, T * w.d * 4, w.E * 4
    total = dict(bytes=0, flops=0, gateup_bytes=0, down_bytes=0, route_bytes=0,
                 gateup_flops=0, down_flops=0, active=[])
    for counts in counts_per_layer:
        act = int((np.asarray(counts) > 0).sum())
        total["active"].append(act)
        total["route_bytes"] += x_b + wr_b + b_b
        total["gateup_bytes"] += act * gu_w + x_b
        total["down_bytes"] += act * dn_w + out_b
        total["gateup_flops"] += 2 * T * w.k * 2 * w.d * w.F
        total["down_flops"] += 2 * T * w.k * w.d * w.F
        total["bytes"] += act * per_w + x_b + wr_b + out_b + b_b
        total["flops"] += 2 * T * w.d * w.E + 2 * T * w.k * 3 * w.d * w.F
    return total


def expert_kernel_names(w, T, num_sms):
    """Which kernels moe_forward's AUTO path runs for this workload (mirrors
    the library's selection: grouped GEMMs from 64 rows per expert on average
    and T >= 512 for bf16 / Q8_0 weights with d % 256 == 0 and F % 128 == 0;
    tensor-core decode for bf16 and affine 4-bit layers with d, F multiples of
    128 and T*k <= 8192 -- one clustered routing+grouping kernel for T <= 128
    (which also writes the grouped fp16 rows of 4-bit layers of up to 16
    tokens; beyond that a gather kernel does), then for bf16
    one persistent kernel for gate/up, SwiGLU, down and the combine when k <= 2
    and the batch has half a wave of whole-K gate/up items of at most 512 KB,
    else the gate/up and down kernels, each in cluster mode for small bf16
    batches (K splits reduced on chip) or with its split-K reduction kernel;
    otherwise the CUDA-core decode kernels), and how many of the library's kernels one
    layer launches.  "fused": the gate/up and down GEMMs run in one kernel,
    timed as one stage."""
    rows = T * w.k
    act16 = w.act_dtype == 1
    if (act16 and w.w_dtype in (1, 2, 3, 4, 5, 6) and w.d % 256 == 0 and w.F % 128 == 0
            and rows >= 64 * w.E and T >= 512):
        q = {1: "bf16", 2: "Q8_0, CTA pairs", 3: "4-bit, CTA pairs", 4: "Q4_K, CTA pairs",
             5: "Q6_K, CTA pairs", 6: "fp8, CTA pairs"}[w.w_dtype]
        return {"file": "tc_gemm.cu", "gateup": f"grouped_gemm_kernel<GATEUP, {q}>",
                "down": f"grouped_gemm_kernel<DOWN, {q}>", "launches": 4, "fused": False}
    if act16 and w.w_dtype in (1, 2, 3, 4, 5, 6) and w.d % 128 == 0 and w.F % 128 == 0 and rows <= 8192:
        n_exp = min(w.E, rows)
        small = T <= 128 and w.d // 64 <= 64 and w.k <= w.E
        q4 = w.w_dtype in (2, 3, 4, 5, 6)   # converted weights (4- or 8-bit): fp16 token rows
        if (not q4 and w.k <= 2 and n_exp * (w.F // 128) * 2 >= 2 * num_sms
                and 2 * 128 * w.d * 2 <= 512 << 10):
            name = "decode_fused_kernel (gate/up + SwiGLU + down + combine, one launch)"
            return {"file": "decode_fused.cu", "gateup": name, "down": name, "fused": True,
                    "launches": (1 if small else 2) + 1}
        fused = 192 <= n_exp * (w.F // 128) <= 2 * num_sms
        direct = w.k <= 2 and n_exp * (w.d // 128) >= 192

        # cluster mode: CS CTAs per unit of 16-row chunks when that fills
        # at most one wave and every K split keeps two k-blocks
        def cluster(units, kb_total):
            for cs in (8, 4, 2):
                if units * cs <= 2 * num_sms and kb_total // cs >= 2:
                    return cs
            return 0
        chunks_cl = n_exp + rows // 16
        cl_gu = 0 if fused else cluster(chunks_cl * (w.F // 128), w.d // 64)
        cl_d = 0 if w.k > 2 or direct else cluster(chunks_cl * (w.d // 128), w.F // 64)
        # 4-bit: the grouped fp16 rows come from the clustered router up to 16
        # tokens, else from a gather kernel
        launches = (1 if small else 2) + (1 if q4 and small and T > 16 else 0) + \
            (1 if fused or cl_gu else 2) + (1 if direct or cl_d else 2)
        tag = {2: ", Q8_0", 3: ", 4-bit", 4: ", Q4_K", 5: ", Q6_K", 6: ", fp8"}.get(w.w_dtype, "")
        gu = f"decode_tc_kernel<GATEUP{tag}> (whole K, writes h)" if fused else \
            f"decode_tc_kernel<GATEUP{tag}> (clusters of {cl_gu}, writes h)" if cl_gu else \
            f"decode_tc_kernel<GATEUP{tag}> + swiglu_reduce_kernel"
        dn = f"decode_tc_kernel<DOWN{tag}> (whole K, adds into out)" if direct else \
            f"decode_tc_kernel<DOWN{tag}> (clusters of {cl_d}, writes out)" if cl_d else \
            f"decode_tc_kernel<DOWN{tag}> + combine_kernel"
        return {"file": "decode_tc.cu", "gateup": gu, "down": dn, "launches": launches,
                "fused": False}
    return {"file": "decode.cu", "gateup": "decode_gateup_kernel", "down": "decode_down_kernel",
            "launches": 4, "fused": False}


def profile_traffic(kernel_key):
    """dram bytes per launch recorded from an ncu capture of this kernel on this
    workload (key "file:stage:workload:T<tokens>"), if the kernel source it was
    taken on is unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel_key:
            rec = {"bytes": float(parts[1]), "sha": parts[2]}
    if not rec:
        return None
    src = os.path.join(ROOT, "expert_routed_ffn_selectedsoftmax_gb300", "csrc",
                       kernel_key.split(":")[0])
    if not os.path.exists(src):
        return None
    return rec["bytes"] if code_sha(open(src).read()) == rec["sha"] else None


def code_sha(text):
    """sha256[:16] of a C/CUDA source with comments and whitespace removed, so
    that a recorded capture stays valid across comment-only edits (string
    literals, e.g. inline PTX, are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch == '"':                               # string literal: copy through
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    code = "".join(out).split()
    return hashlib.sha256(" ".join(code).encode()).hexdigest()[:16]


# ------------------------------------------------------------- CPU oracle
def oracle_runs(layer, rows, runs=3, mode=0):
    """Time the oracle `runs` times on token rows `rows` of a host layer (all
    host cores); returns (tokens/s of each run, threads)."""
    import copy
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    sub = copy.copy(layer)
    sub.x = np.ascontiguousarray(layer.x[rows])
    sub.T = len(rows)
    rates = []
    for _ in range(runs):
        t0 = time.perf_counter()
        oracle.moe_forward(sub, nthreads=threads, mode=mode)
        rates.append(sub.T / (time.perf_counter() - t0))
    return rates, threads


def oracle_baseline(layers_host, sample_rows, mode=0, runs=3):
    """The oracle's tokens/s on the host cores: the median of `runs` timed
    passes, each over the first `sample_rows` token rows of every given host
    layer (whole layers when sample_rows >= T)."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    per_run = []
    for _ in range(runs):
        tok, secs = 0, 0.0
        for layer in layers_host:
            rates, _ = oracle_runs(layer, np.arange(min(sample_rows, layer.T)), runs=1, mode=mode)
            n = min(sample_rows, layer.T)
            tok += n
            secs += n / rates[0]
        per_run.append(tok / secs)
    return {"value": statistics.median(per_run), "runs": per_run, "unit": "tokens/s",
            "cores": threads, "kind": "oracle", "cpu_model": host_cpu_model()}


def host_layer_from_device(w, dl, T):
    """A workloads.Layer (host storage arrays) from one device-drawn layer."""
    import torch
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl

    def bits(t):
        if t.dtype == torch.float32:
            return t.contiguous().cpu().numpy()
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    if w.w_dtype in (wl.Q8_0, wl.Q4_A64, wl.Q4_K, wl.Q6_K, wl.FP8):   # the oracle reads the blocks themselves
        wts = {n: dl["blocks"][n].cpu().numpy() for n in ("w_gate", "w_up", "w_down")}
    else:
        wts = {n: bits(dl[n]) for n in ("w_gate", "w_up", "w_down")}
    return wl.Layer(T=T, d=w.d, E=w.E, k=w.k, F=w.F, act_dtype=w.act_dtype, w_dtype=w.w_dtype,
                    x=bits(dl["x"]), w_router=bits(dl["w_router"]),
                    bias=dl["bias"].float().cpu().numpy(), **wts)


def host_cpu_model():
    """The host CPU's model name (x86: /proc/cpuinfo; Arm: lscpu), for the CPU baseline."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def percentiles(samples_ms):
    """p10 / median / p90 of per-step times (nearest rank)."""
    v = sorted(samples_ms)
    at = lambda q: v[min(len(v) - 1, max(0, int(math.ceil(q * len(v))) - 1))]
    return {"p10": at(0.10), "median": statistics.median(v), "p90": at(0.90), "n": len(v)}


def run_reference(args, w, T, layers):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import oracle
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    oracle.build()
    threads = oracle.default_threads()
    # host-drawn layer of the same shapes and distributions; each step runs the
    # oracle on a bounded sample of `sample_T` tokens of that layer
    layer = wl.make_layer(w, seed=0, T=T)
    sample_T = min(T, max(1, threads))
    import copy
    subs = []
    for s in range(4):
        sub = copy.copy(layer)
        rows = (np.arange(sample_T) + s * sample_T) % T
        sub.x = np.ascontiguousarray(layer.x[rows])
        sub.T = sample_T
        subs.append(sub)
    for i in range(args.warmup):
        oracle.moe_forward(subs[i % 4], nthreads=threads, mode=scoring_mode(args))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.moe_forward(subs[i % 4], nthreads=threads, mode=scoring_mode(args))
    dt = time.perf_counter() - t0
    value = sample_T * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, T, layers, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "cpu_model": host_cpu_model(),
                         "sample": f"{sample_T} tokens of one {w.name} layer per step "
                                   f"(fp64 C oracle, {threads} threads)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, T, layers, args):
    return {"workload": w.name, "T": T, "d": w.d, "E": w.E, "k": w.k, "F": w.F,
            "layers": layers, "act_dtype": "bf16" if w.act_dtype else "f32",
            "w_dtype": {0: "f32", 1: "bf16", 2: "q8_0", 3: "q4_a64", 4: "q4_k", 5: "q6_k", 6: "fp8_e4m3"}[w.w_dtype],
            "bias": w.bias, "global_batch": T * max(1, args.gpus), "parallelism": "replicas",
            "l2": "inputs larger than L2: every step reads all layers' expert weights",
            "graph": not args.no_graph, "scoring": args.scoring,
            "dense": bool(args.dense)}


def dtype_label(w, names):
    """The arithmetic the path runs in: the storage of the expert weights and,
    for quantised weights, whether the CUDA-core kernels (fp32) or the
    tensor-core kernels (fp16 operands) run them."""
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    if w.w_dtype in (wl.F32, wl.BF16):
        return {wl.F32: "f32", wl.BF16: "bf16"}[w.w_dtype]
    fmt = {wl.Q8_0: "q8_0", wl.Q4_A64: "affine 4-bit", wl.Q4_K: "q4_k", wl.Q6_K: "q6_k",
           wl.FP8: "fp8 e4m3"}[w.w_dtype]
    how = "f32 CUDA-core arithmetic" if names["file"] == "decode.cu" else "f16 tensor-core operands"
    return f"{fmt} weights, {how}"


def scoring_mode(args):
    """moe_forward scoring argument (and the oracle's mode) for --scoring."""
    return {"selected_softmax": 0, "softmax": 1, "sigmoid": 2}[args.scoring]


def compute_peak(w, peaks, dev_props, kernels=None):
    """The compute roofline of a workload's expert arithmetic: the measured
    dense bf16 tensor peak for bf16 weights and for block-quantised weights on
    the tensor-core kernels (fp16 operands, the same dense rate); for fp32
    weights and block-quantised weights on the CUDA-core kernels, which run as
    fp32 FMAs, 128 FMA lanes x 2 flops per SM per clock at the device's
    maximum SM clock ("alu")."""
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    simt = kernels is None or kernels["file"] == "decode.cu"
    if w.w_dtype == wl.F32 or (w.w_dtype in (wl.Q8_0, wl.Q4_A64, wl.Q4_K, wl.Q6_K, wl.FP8) and simt):
        mhz = float(peaks.get("sm_max_mhz") or 0) or dev_props.clock_rate / 1e3
        return dev_props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12, "alu", \
            "fp32 FMA: SMs x 128 lanes x 2 flops x max SM clock"
    return peak_value(peaks, "bf16_tflops"), "tensor", "bf16_tflops"


ZIPF_FIXTURE = os.path.join(ROOT, "tests", "golden", "zipf_bias_zonos3_mini_prefill.txt")


def zipf_fit(w, T, layers):
    """The fitted selection biases and Zipf targets of a full-size Zipf
    workload (tests/golden/zipf_bias_zonos3_mini_prefill.txt, written with
    the oracle's routing on the layers' host-drawn inputs), or None."""
    if w.bias != "zipf" or w.name != "zonos3_mini_prefill" or (T is not None and T != w.T) \
            or not os.path.exists(ZIPF_FIXTURE):
        return None
    rec = {}
    for line in open(ZIPF_FIXTURE):
        if line.startswith("#") or not line.strip():
            continue
        key, layer, *vals = line.split()
        rec.setdefault(int(layer), {})[key] = np.array([float(v) for v in vals])
    if any(i not in rec for i in range(layers)):
        return None
    return [rec[i]["bias"].astype(np.float32) for i in range(layers)], \
        [rec[i]["target"] for i in range(layers)]


def zipf_report(targets, counts_per_layer):
    """Achieved loads (the layer's own routing, read back) against the Zipf
    targets: head share, tail, and the fraction of assignments off target."""
    out = []
    for tgt, cnt in zip(targets, counts_per_layer):
        cnt = np.asarray(cnt, dtype=np.float64)
        order = np.argsort(-tgt)
        out.append({"top_share": float(cnt[order[0]] / cnt.sum()),
                    "top_share_target": float(tgt[order[0]] / tgt.sum()),
                    "bottom_rows": int(cnt[order[-1]]), "bottom_rows_target": float(tgt[order[-1]]),
                    "off_target_frac": float(np.abs(cnt - tgt).sum() / cnt.sum())})
    return out


def setup_stack(pkg, wl, w, T, layers, seed, dev):
    """Device stack of `layers` layers of workload w (block-quantised weights
    repacked once), plus the dtypes moe_forward takes.  A full-size Zipf
    workload takes its fitted biases and the inputs they were fitted on."""
    import torch
    fit = zipf_fit(w, T, layers)
    stack = wl.make_device_stack(w, seed=seed, layers=layers, T=T, device=dev,
                                 zipf_biases=fit[0] if fit else None)
    act_dt = pkg.MOE_F32 if w.act_dtype == wl.F32 else pkg.MOE_BF16
    w_dt = {wl.F32: pkg.MOE_F32, wl.BF16: pkg.MOE_BF16, wl.Q8_0: pkg.MOE_Q8_0,
            wl.Q4_A64: pkg.MOE_Q4_A64, wl.Q4_K: pkg.MOE_Q4_K, wl.Q6_K: pkg.MOE_Q6_K,
            wl.FP8: pkg.MOE_FP8}[w.w_dtype]
    if w_dt in (pkg.MOE_Q8_0, pkg.MOE_Q4_A64, pkg.MOE_Q4_K, pkg.MOE_Q6_K, pkg.MOE_FP8):
        pack = {pkg.MOE_Q8_0: pkg.moe_pack_q8_0, pkg.MOE_Q4_A64: pkg.moe_pack_q4_a64,
                pkg.MOE_Q4_K: pkg.moe_pack_q4_k, pkg.MOE_Q6_K: pkg.moe_pack_q6_k,
                pkg.MOE_FP8: pkg.moe_pack_fp8}[w_dt]
        for L in stack:
            L["blocks"] = {n: L[n] for n in ("w_gate", "w_up", "w_down")}
            for n, rows, cols in (("w_gate", w.E * w.F, w.d), ("w_up", w.E * w.F, w.d),
                                  ("w_down", w.E * w.d, w.F)):
                L[n] = pack(L[n].reshape(-1), rows, cols)
    # the stack was drawn on the current stream; the layer calls run on the
    # runner's own stream
    torch.cuda.synchronize(dev)
    return stack, act_dt, w_dt


class Runner:
    """One workload's stack on the device and the layer calls a step makes."""

    def __init__(self, pkg, wl, w, T, layers, seed, dev, scoring=0, dense=False):
        import torch
        self.pkg, self.w, self.T, self.layers, self.dev = pkg, w, T, layers, dev
        self.scoring, self.dense = scoring, dense
        self.stack, self.act_dt, self.w_dt = setup_stack(pkg, wl, w, T, layers, seed, dev)
        self.ws_bytes = pkg.moe_workspace_size(T, w.d, w.E, w.k, w.F, self.act_dt, self.w_dt)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.outs = [torch.empty((T, w.d), dtype=torch.float32, device=dev) for _ in range(layers)]
        self.stream = torch.cuda.Stream(device=dev)
        self.graph = None

    def layer_call(self, i, events=None, x=None):
        L, w, pkg = self.stack[i], self.w, self.pkg
        x = L["x"] if x is None else x
        if self.dense and events is None:
            pkg.moe_ffn_dense(x, L["w_gate"], L["w_up"], L["w_down"], F=w.F, w_dtype=self.w_dt,
                              out=self.outs[i], workspace=self.ws)
            return
        # (dense layers: the per-stage timings come from the same one-expert
        # layer through moe_forward_profiled -- same expert kernels)
        pkg.moe_forward(x, L["w_router"], L["bias"], L["w_gate"], L["w_up"], L["w_down"],
                        w.k, F=w.F, w_dtype=self.w_dt, out=self.outs[i], workspace=self.ws,
                        events=events, scoring=self.scoring)

    def step(self):
        for i in range(self.layers):
            self.layer_call(i)

    def counts_per_layer(self):
        """Per-expert row counts each layer's own routing produced (read back
        from the workspace after the layer ran)."""
        import torch
        out = []
        with torch.cuda.stream(self.stream):
            for i in range(self.layers):
                self.layer_call(i)
                self.stream.synchronize()
                r = self.pkg.read_routing(self.ws, self.T, self.w.d, self.w.E, self.w.k, self.w.F,
                                          self.act_dt, self.w_dt)
                out.append(r["counts"].cpu().numpy().copy())
        return out

    def capture(self, warmup, graph=True):
        import torch
        with torch.cuda.stream(self.stream):
            for _ in range(max(3, warmup)):
                self.step()
        self.stream.synchronize()
        if graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self.step()
            with torch.cuda.stream(self.stream):
                for _ in range(3):
                    self.graph.replay()
            self.stream.synchronize()
        assert self.pkg.moe_check(self.ws) == 0

    def replay(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.step()

    def time_steps(self, steps):
        """Device time of `steps` back-to-back steps (ms), CUDA events on the
        launching stream."""
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                self.replay()
            e1.record(self.stream)
        self.stream.synchronize()
        return e0.elapsed_time(e1)

    def stage_us(self, n_prof):
        """Per-launch µs of each stage (route, permute, gather, gate/up, down):
        the same layers with caller events at the stage boundaries."""
        import torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)]
               for _ in range(self.layers)]
        # torch only reports elapsed time for events it has recorded itself once;
        # the library re-records the same events at its stage boundaries
        for row in evs:
            for ev in row:
                ev.record(self.stream)
        self.stream.synchronize()
        stage_ms = np.zeros(5)
        with torch.cuda.stream(self.stream):
            for _ in range(n_prof):
                for i in range(self.layers):
                    self.layer_call(i, events=evs[i])
                self.stream.synchronize()
                for i in range(self.layers):
                    for s in range(5):
                        stage_ms[s] += evs[i][s].elapsed_time(evs[i][s + 1])
        return stage_ms / (n_prof * self.layers) * 1e3

    def free(self):
        self.stack = self.outs = self.ws = self.graph = None


STAGES = ["route", "permute", "gather", "gateup", "down"]


def roofline_of(w, T, layers, alg, stage_us, names, peaks, peak_src, dev_props, dense=False):
    """Roofline object of the dominant expert kernel (the slower of gate/up and
    down by live stage events): its algorithmic bytes (or flops, past the
    ridge) per launch over its measured duration."""
    hbm = peak_value(peaks, "hbm_gbs")
    cpeak, cbound, csrc = compute_peak(w, peaks, dev_props, names)
    if names.get("fused"):
        # one kernel streams both GEMMs' weights: its stage is the gate/up one
        dominant, dom_us = "fused", stage_us[3]
        names = dict(names, fused=names["gateup"])
        dom_bytes = (alg["gateup_bytes"] + alg["down_bytes"]) / layers
        dom_flops = (alg["gateup_flops"] + alg["down_flops"]) / layers
    else:
        dominant = "gateup" if stage_us[3] >= stage_us[4] else "down"
        dom_us = stage_us[3] if dominant == "gateup" else stage_us[4]
        dom_bytes = alg[f"{dominant}_bytes"] / layers
        dom_flops = alg[f"{dominant}_flops"] / layers
    compute_bound = dom_flops / dom_bytes > cpeak * 1e12 / (hbm * 1e9)
    traffic = profile_traffic(f"{names['file']}:{dominant}:{w.name}{'-dense' if dense else ''}:T{T}")
    if compute_bound:
        achieved = dom_flops / (dom_us * 1e-6) / 1e12
        return {"bound": cbound, "kernel": names[dominant], "achieved": achieved,
                "peak": cpeak, "unit": "TFLOP/s", "frac": achieved / cpeak, "traffic": traffic,
                "peak_source": f"{csrc} of {peak_src}" if cbound == "tensor" else csrc,
                "flops_per_launch": dom_flops, "bytes_per_launch": dom_bytes,
                "us_per_launch": dom_us}
    achieved = dom_bytes / (dom_us * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": names[dominant], "achieved": achieved, "peak": hbm,
            "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
            "peak_source": f"hbm_gbs of {peak_src}", "bytes_per_launch": dom_bytes,
            "flops_per_launch": dom_flops, "us_per_launch": dom_us}


def layer_stats(w, alg, ms_per_step, layers, peaks, dev_props, stage_us, names=None):
    hbm = peak_value(peaks, "hbm_gbs")
    cpeak, cbound, _ = compute_peak(w, peaks, dev_props, names)
    gbs = alg["bytes"] / (ms_per_step * 1e-3) / 1e9
    return {"us_per_layer": ms_per_step * 1e3 / layers, "algorithmic_GBps": gbs,
            "TFLOPS": alg["flops"] / (ms_per_step * 1e-3) / 1e12, "frac_hbm": gbs / hbm,
            "roofline_frac": layer_roofline_frac(alg["bytes"], alg["flops"], ms_per_step * 1e-3,
                                                 hbm, cpeak),
            "compute_peak": {"value": cpeak, "unit": "TFLOP/s", "kind": cbound},
            "bytes_per_step": alg["bytes"], "flops_per_step": alg["flops"],
            "active_experts_per_layer": alg["active"],
            "stage_us": dict(zip(STAGES, [round(float(v), 3) for v in stage_us]))}


# The configurations every default run measures beside the headline workload
# (each at N = 1 on rank 0's GPU, the oracle beside it): (workload, T,
# layers, oracle token sample per layer).
SIDE_WORKLOADS = [("tiny_fp32", None, None, 8), ("zonos2_decode", 1, None, 1),
                  ("zonos2_decode", 8, None, 8), ("zonos2_decode", 64, None, 64),
                  ("zonos3_mini_prefill", None, None, 512), ("zonos2_prefill_q8", None, None, 192),
                  ("zonos2_decode_q4", 1, None, 1), ("zonos2_decode_q4", 8, None, 8),
                  ("zonos2_decode_q4", 64, None, 64), ("zonos2_prefill_q4", None, None, 192),
                  ("zonos2_decode_q4k", 1, None, 1), ("zonos2_decode_q4k", 8, None, 8),
                  ("zonos2_decode_q4k", 64, None, 64), ("zonos2_prefill_q4k", None, None, 192),
                  ("zonos2_decode_q8", 1, None, 1), ("zonos2_decode_q8", 8, None, 8),
                  ("zonos2_decode_q8", 64, None, 64),
                  ("zonos2_decode_q6k", 1, None, 1), ("zonos2_decode_q6k", 8, None, 8),
                  ("zonos2_decode_q6k", 64, None, 64), ("zonos2_prefill_q6k", None, None, 192),
                  ("zonos2_decode_fp8", 1, None, 1), ("zonos2_decode_fp8", 8, None, 8),
                  ("zonos2_decode_fp8", 64, None, 64), ("zonos2_prefill_fp8", None, None, 192)]


def measure_side_workload(pkg, wl, name, T, layers, sample_rows, dev, peaks, peak_src,
                          dev_props, target_s=0.3, with_oracle=True):
    """One configuration measured on its own: graph replays of its stack timed
    with events, stage events, the layer and dominant-kernel roofline
    fractions, and the oracle's tokens/s on the host cores (median of 3)."""
    import torch
    w = wl.WORKLOADS[name]
    T = w.T if T is None else T
    layers = w.layers if layers is None else layers
    def note(what):
        print(f"[side {name} T={T}] {what}", file=sys.stderr, flush=True)
    r = Runner(pkg, wl, w, T, layers, seed=11, dev=dev)
    note("stack ready")
    counts = r.counts_per_layer()
    note("routing read back")
    alg = algorithmic(w, T, counts)
    r.capture(3)
    note("warm-up and graph done")
    est = r.time_steps(3) / 3
    steps = int(min(2000, max(20, math.ceil(target_s * 1e3 / max(est, 1e-3)))))
    t_ms = r.time_steps(steps)
    ms = t_ms / steps
    stage = r.stage_us(max(5, min(50, steps // 4)))
    names = expert_kernel_names(w, T, dev_props.multi_processor_count)
    res = {"workload": name, "T": T, "d": w.d, "E": w.E, "k": w.k, "F": w.F,
           "w_dtype": wl.DTYPE_NAMES[w.w_dtype], "layers": layers, "steps": steps,
           "ms_per_step": ms, "tokens_per_s": T * layers / (ms * 1e-3),
           "layer": layer_stats(w, alg, ms, layers, peaks, dev_props, stage, names),
           "roofline": roofline_of(w, T, layers, alg, stage, names, peaks, peak_src, dev_props),
           "gpu_launches_per_layer": names["launches"]}
    fit = zipf_fit(w, T, layers)
    if fit:   # the fitted Zipf loads, as this run's own routing produced them
        res["zipf_loads"] = zipf_report(fit[1], counts)
    if with_oracle:
        host = host_layer_from_device(w, r.stack[0], T)
        res["cpu_baseline"] = oracle_baseline([host], sample_rows)
        res["cpu_baseline"]["sample"] = (f"median of 3 passes over {min(sample_rows, T)} of the "
                                         f"{T} tokens of one layer (fp64 C oracle)")
    r.free()
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def run_side_child(name, T, no_cpu_baseline):
    """Measure one configuration in a child process (bench.py --side NAME[:T]);
    its JSON result, or a record of the failure."""
    cmd = [sys.executable, os.path.abspath(__file__), "--side", f"{name}:{T if T else ''}"]
    if no_cpu_baseline:
        cmd.append("--no-cpu-baseline")
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    except subprocess.TimeoutExpired:
        return {"workload": name, "T": T, "error": "timed out after 600 s"}
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if r.returncode != 0 or not lines:
        tail = (r.stderr or r.stdout)[-400:]
        return {"workload": name, "T": T, "error": f"exit {r.returncode}: {tail}"}
    return json.loads(lines[-1])


def side_main(args):
    """bench.py --side NAME[:T]: one configuration of SIDE_WORKLOADS, alone."""
    import torch
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    name, _, t = args.side.partition(":")
    T = int(t) if t else None
    rows = next((r for n, sT, _, r in SIDE_WORKLOADS if n == name and sT == T), 64)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    pkg.load_library()
    peaks, peak_src = load_peaks()
    res = measure_side_workload(pkg, wl, name, T, None, rows, dev, peaks, peak_src,
                                torch.cuda.get_device_properties(dev),
                                with_oracle=not args.no_cpu_baseline)
    print(json.dumps(res), flush=True)
    return 0


def main():
    args = parse()
    if args.side:
        return side_main(args)
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    if args.dense:   # one expert of the workload's shape, no router
        import dataclasses
        w = dataclasses.replace(w, E=1, k=1)
    T = args.T if args.T is not None else w.T
    layers = args.layers if args.layers is not None else w.layers
    if args.impl == "reference":
        return run_reference(args, w, T, layers)

    import torch
    import expert_routed_ffn_selectedsoftmax_gb300 as pkg
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pkg.load_library()
    dev_props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()

    # ------------------------------------------------------------ inputs
    run = Runner(pkg, wl, w, T, layers, seed=1 + rank, dev=dev, scoring=scoring_mode(args),
                 dense=args.dense)
    stack, w_dt, stream = run.stack, run.w_dt, run.stream
    counts_per_layer = run.counts_per_layer()
    alg = algorithmic(w, T, counts_per_layer)

    # --------------------------------------------------------- warm-up + graph
    run.capture(args.warmup, graph=not args.no_graph)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ------------------------------------------------------------ timed region
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    t_ms = run.time_steps(args.steps)
    clk = clocks.stop()
    barrier()
    t_ms = max_over_ranks(t_ms, world, dev)
    ms_per_step = t_ms / args.steps
    tokens_per_step = T * layers
    value = job_throughput(tokens_per_step, world, ms_per_step)

    # -------------------------------- per-step distribution (separate pass)
    # one event between consecutive steps; the contract's number above is
    # the bracketed total, this only adds its spread
    n_dist = max(1, min(args.steps, 200))
    step_evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_dist + 1)]
    with torch.cuda.stream(stream):
        step_evs[0].record(stream)
        for i in range(n_dist):
            run.replay()
            step_evs[i + 1].record(stream)
    stream.synchronize()
    step_dist = percentiles([step_evs[i].elapsed_time(step_evs[i + 1]) for i in range(n_dist)])

    # --------------------------------------------- per-kernel (stage) timing
    stage_us = run.stage_us(max(1, min(args.steps, 200)))
    names = expert_kernel_names(w, T, dev_props.multi_processor_count)
    roofline = roofline_of(w, T, layers, alg, stage_us, names, peaks, peak_src, dev_props,
                           dense=args.dense)

    # ------------------------------------------------------------- e2e
    # through the public API with host buffers: pinned x in, fp32 out back, per step
    outs, ws = run.outs, run.ws
    hx = [L["x"].cpu().pin_memory() for L in stack]
    hout = [torch.empty((T, w.d), dtype=torch.float32).pin_memory() for _ in range(layers)]
    dx = [torch.empty_like(L["x"]) for L in stack]
    n_e2e = max(1, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_layer(i):
        L = stack[i]
        if args.dense:
            pkg.moe_ffn_dense(dx[i], L["w_gate"], L["w_up"], L["w_down"], F=w.F,
                              w_dtype=w_dt, out=outs[i], workspace=ws)
        else:
            pkg.moe_forward(dx[i], L["w_router"], L["bias"], L["w_gate"], L["w_up"],
                            L["w_down"], w.k, F=w.F, w_dtype=w_dt, out=outs[i],
                            workspace=ws, scoring=scoring_mode(args))

    def e2e_serial():
        """Every copy and layer in order on one stream."""
        def one_step():
            for i in range(layers):
                dx[i].copy_(hx[i], non_blocking=True)
            for i in range(layers):
                e2e_layer(i)
            for i in range(layers):
                hout[i].copy_(outs[i], non_blocking=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                one_step()
        stream.synchronize()
        barrier()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_e2e):
                one_step()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / n_e2e

    def e2e_pipelined():
        """Copies on two copy streams: the host-to-device copy of layer i+1 and
        the device-to-host copy of layer i-1 run while layer i computes.  Layer
        i waits for its input copy and for the previous step's read-back of
        out[i]; the input copy of the next step waits for layer i to finish
        reading x[i].  The timed region ends after the last read-back."""
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(layers)]     # x[i] on the device
        ev_done = [torch.cuda.Event() for _ in range(layers)]   # layer i computed
        ev_back = [torch.cuda.Event() for _ in range(layers)]   # out[i] read back
        state = {"first": True}

        def one_step():
            first = state["first"]
            for i in range(layers):
                with torch.cuda.stream(h2d_s):
                    if not first:
                        h2d_s.wait_event(ev_done[i])
                    dx[i].copy_(hx[i], non_blocking=True)
                    ev_in[i].record(h2d_s)
                with torch.cuda.stream(stream):
                    stream.wait_event(ev_in[i])
                    if not first:
                        stream.wait_event(ev_back[i])
                    e2e_layer(i)
                    ev_done[i].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_done[i])
                    hout[i].copy_(outs[i], non_blocking=True)
                    ev_back[i].record(d2h_s)
            state["first"] = False

        for _ in range(3):
            one_step()
        torch.cuda.synchronize(dev)
        barrier()
        e0.record(stream)
        h2d_s.wait_event(e0)
        for _ in range(n_e2e):
            one_step()
        for i in range(layers):
            stream.wait_event(ev_back[i])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n_e2e

    # both schedules are timed and the faster is reported (with few layers the
    # cross-stream event hops cost more than the copies they hide)
    serial_ms = e2e_serial()
    try:
        overlap_ms = e2e_pipelined()
    except Exception as exc:   # the serial measurement stands if stream pipelining fails
        torch.cuda.synchronize(dev)
        overlap_ms, overlap_err = None, str(exc)[:120]
    else:
        overlap_err = None
    if overlap_ms is not None and overlap_ms < serial_ms:
        e2e_ms, e2e_mode = overlap_ms, "copies overlapped with compute (faster here)"
    else:
        e2e_ms, e2e_mode = serial_ms, "serial (faster here)" if overlap_err is None else \
            f"serial (overlap failed: {overlap_err})"
    e2e_alt = {"serial_tokens_per_s": tokens_per_step * world / (serial_ms * 1e-3),
               "overlapped_tokens_per_s": None if overlap_ms is None
               else tokens_per_step * world / (overlap_ms * 1e-3)}
    e2e_value = tokens_per_step * world / (e2e_ms * 1e-3)
    h2d = sum(t.numel() * t.element_size() for t in hx)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    # ------------------------------------------------------- CPU baseline
    cpu = None
    host_layers = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_layers = [host_layer_from_device(w, stack[i], T) for i in range(layers)]
    run.free()
    del stack, outs, ws, hx, hout, dx
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    if host_layers is not None:
        cpu = oracle_baseline(host_layers, T, mode=scoring_mode(args))
        cpu["sample"] = (f"median of 3 passes over all {layers} layers of one step, all {T} "
                         f"tokens each (fp64 C oracle, {cpu['cores']} threads)")

    # ------------------------------- every other configuration, measured alone
    # (each in a process of its own on this GPU, after this process's own
    # measurement is complete: its stacks get the device to themselves, and a
    # failure there cannot take the headline line with it)
    side = None
    if world == 1 and not args.no_workloads and args.workload == "zonos3_mini_decode" and \
            not args.dense and args.T is None and args.layers is None and args.scoring == \
            "selected_softmax":
        side = [run_side_child(name, sT, args.no_cpu_baseline) for name, sT, _, _ in SIDE_WORKLOADS]

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_label(w, names),
        "data": "synthetic", "config": config_dict(w, T, layers, args),
        "clocks": clk, "e2e": {"value": e2e_value, "unit": "tokens/s", "mode": e2e_mode, **e2e_alt,
                               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": names["launches"] * layers * args.steps,
        "roofline": roofline, "cpu_baseline": cpu, "step_ms": step_dist,
        "layer": layer_stats(w, alg, ms_per_step, layers, peaks, dev_props, stage_us, names),
        "workloads": side,
        "zipf_loads": (zipf_report(zipf_fit(w, T, layers)[1], counts_per_layer)
                       if zipf_fit(w, T, layers) else None),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
