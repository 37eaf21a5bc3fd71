"""Host-side checks of the benchmark's multi-rank logic and of its reference
arm (no GPU): two gloo ranks on CPU take the slowest rank's time, whole-job
throughput counts every rank's tokens, and `bench.py --impl reference` prints
one JSON line with the contract's keys on rank 0 and nothing on other ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    times = [3.25, 5.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), times, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert got == [5.5, 5.5]


def test_single_rank_and_throughput():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    # 128 tokens x 10 layers per rank per step, 2 ranks, 0.5 ms per step
    assert bench.job_throughput(1280, 2, 0.5) == pytest.approx(5.12e6)


def test_layer_roofline_fraction_takes_the_slower_bound():
    sys.path.insert(0, ROOT)
    import bench
    # 6.8 GB at 6.8 TB/s = 1 ms; 1.9 TFLOP at 1.9 PF = 1 ms; measured 2 ms -> 0.5
    assert bench.layer_roofline_frac(6.8e9, 1.9e12, 2e-3, 6800.0, 1900.0) == pytest.approx(0.5)
    # bytes-bound: flops negligible
    assert bench.layer_roofline_frac(6.8e9, 1.0, 4e-3, 6800.0, 1900.0) == pytest.approx(0.25)
    # flops-bound: 3.8 TFLOP = 2 ms at peak, measured 2.5 ms
    assert bench.layer_roofline_frac(1.0, 3.8e12, 2.5e-3, 6800.0, 1900.0) == pytest.approx(0.8)


def test_step_percentiles_nearest_rank():
    sys.path.insert(0, ROOT)
    import bench
    p = bench.percentiles([float(v) for v in range(10, 0, -1)])   # 1..10, unsorted
    assert p == {"p10": 1.0, "median": 5.5, "p90": 9.0, "n": 10}
    assert bench.percentiles([2.0]) == {"p10": 2.0, "median": 2.0, "p90": 2.0, "n": 1}


def test_traffic_record_survives_comment_edits_only():
    sys.path.insert(0, ROOT)
    import bench
    src = 'int f(int a) { // one\n  return a + 1; /* two */ }\nconst char *s = "a // b";\n'
    same = 'int f(int a) {\n  /* other words */ return a + 1; }  const char *s = "a // b";'
    assert bench.code_sha(src) == bench.code_sha(same)
    assert bench.code_sha(src) != bench.code_sha(src.replace("a + 1", "a + 2"))
    assert bench.code_sha(src) != bench.code_sha(src.replace('"a // b"', '"a // c"'))
    assert bench.profile_traffic("decode_tc.cu:down:no_such_workload:T1") is None


def _reference(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_prints_the_contract_line_on_rank_zero_only():
    lines = _reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert isinstance(j["cpu_baseline"]["cpu_model"], str) and j["cpu_baseline"]["cpu_model"]
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]
    assert j["config"]["workload"] == "tiny_fp32"
    assert _reference({"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_every_workload_has_its_labels_and_peaks():
    """Every workload the benchmark can run (its side configurations and every
    named workload at its own T) gets a config, a kernel selection, a dtype
    label, a compute peak and nonzero expert bytes on the host, so that a new
    weight storage cannot reach the GPU run without them."""
    import argparse
    import types
    sys.path.insert(0, ROOT)
    import bench
    from expert_routed_ffn_selectedsoftmax_gb300 import workloads as wl
    args = argparse.Namespace(gpus=1, no_graph=False, scoring="selected_softmax", dense=False)
    props = types.SimpleNamespace(multi_processor_count=152, clock_rate=2070000)
    peaks = {"hbm_gbs": 6670.9, "bf16_tflops": 1943.5, "sm_max_mhz": 2070}
    cases = [(name, T) for name, T, _, _ in bench.SIDE_WORKLOADS] + [(n, None) for n in wl.WORKLOADS]
    for name, T in cases:
        w = wl.WORKLOADS[name]
        T = w.T if T is None else T
        cfg = bench.config_dict(w, T, w.layers, args)
        assert cfg["workload"] == name and cfg["w_dtype"] == wl.DTYPE_NAMES[w.w_dtype]
        names = bench.expert_kernel_names(w, T, 152)
        assert names["launches"] >= 1 and names["file"] in ("decode.cu", "decode_tc.cu", "decode_fused.cu",
                                                            "tc_gemm.cu")
        assert bench.dtype_label(w, names)
        peak = bench.compute_peak(w, peaks, props, names)
        assert peak[0] > 0
        assert wl.weight_bytes_per_expert(w.d, w.F, w.w_dtype) > 0
