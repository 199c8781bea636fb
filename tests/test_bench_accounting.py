"""The benchmark's byte and FLOP accounting (the numerators of every roofline figure),
checked against hand counts, and the reference arm's JSON line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_attention_09_gb300 import workloads as W  # noqa: E402


def test_cache_bytes_per_token_of_every_format():
    # K and V rows of every kv head, plus two FP32 scales per kv head for coded formats
    assert bench.kv_token_bytes(W.workload("tinyllama-int8")) == 4 * (2 * 64 + 8)
    assert bench.kv_token_bytes(W.workload("tinyllama-fp8")) == 4 * (2 * 64 + 8)
    assert bench.kv_token_bytes(W.workload("tinyllama-int4")) == 4 * (2 * 32 + 8)
    assert bench.kv_token_bytes(W.workload("smollm2-f32")) == 3 * 2 * 64 * 4
    assert bench.kv_token_bytes(W.workload("qwen-bf16")) == 2 * 2 * 128 * 2


def test_decode_bytes_of_the_benchmark_workload():
    wl = W.workload("tinyllama-int8")
    b = wl.batches[0]
    kv = 256 * 1024 * 4 * (2 * 64 + 8)       # every cached token's K, V and scales once
    q = out = 256 * 32 * 64 * 4              # FP32 queries in, FP32 outputs out
    tables = 256 * (1024 // 16) * 4          # the table entries that are read
    lens = 256 * 4
    assert bench.decode_bytes(wl, b) == kv + q + out + tables + lens == 146867200


def test_append_and_prefill_accounting():
    wl = W.workload("mixed")
    T = 4 + 2 * 512                          # one new token per decode sequence + 2 chunks
    assert bench.append_bytes(wl) == T * 2 * 128 * 2 * 2 + T * 2 * (2 * 128 * 2) + T * 4
    pb = [b for b in wl.batches if b.kind == "prefill"][0]
    keys = sum(2048 + i + 1 for i in range(512))  # causal: row i sees prior + i + 1 keys
    assert bench.prefill_flops(wl, pb) == 2 * keys * 4 * 128 * 12


def test_job_rate_is_all_ranks_work_over_the_slowest_time():
    assert bench.job_rate(10.0, 4, 2.0) == 20.0


def test_reference_arm_line(capsys, monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload", "tiny",
                                      "--steps", "3", "--warmup", "3"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    ident = bench.workload_config(W.workload("tiny"))
    assert all(d["config"][k] == v for k, v in ident.items())
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_our_arm_line_assembly(capsys, monkeypatch):
    """The JSON line of our arm, assembled from fixed measurements (the GPU measurement
    itself is replaced): every contract key, the roofline from the decode bytes and time,
    the whole-job value from all bytes of the step."""
    wl = W.workload("tinyllama-int8")
    acc = bench.step_accounting(wl)
    ms = 0.034  # per step
    kern = {"append": {"ms": 0.0026, "replays": 5, "launches_per_graph": 50},
            "decode": {"ms": 0.0308, "replays": 5, "launches_per_graph": 50}}
    e2e = {"value": 1.0, "unit": "GB/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1,
           "ms_per_step": 0.08, "launches": "direct"}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 5, "reasons": []}
    table = {"tinyllama-int8": bench.workload_entry(wl, acc, kern, 6794.5, (1903.5, 1700.2, "m"))}
    monkeypatch.setattr(bench, "run_ours", lambda args, rank, world: dict(
        wl=wl, acc=acc, R=4, ms=ms, kern=kern, clocks=clocks, e2e=e2e, fused=False, n_append=256,
        workloads=table))
    monkeypatch.setattr(bench, "measured_hbm", lambda: (6794.5, "measured"))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--no-cpu-baseline", "--steps", "7",
                                      "--warmup", "3"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 7 and d["gpu_launches"] == 7 * 2
    assert abs(d["value"] - acc["total"] / (ms * 1e-3) / 1e9) < 0.01
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["peak"] == 6794.5 and r["unit"] == "GB/s"
    assert abs(r["achieved"] - acc["decode"] / (0.0308e-3) / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6794.5) < 1e-3
    assert r["algorithmic_bytes_per_launch"] == acc["decode"]
    assert d["config"]["workload"] == "tinyllama-int8" and d["config"]["layers"] == 1
    assert d["dtype"] == "int8-kv/f32-acc"
    w = d["workloads"]["tinyllama-int8"]["decode"]
    assert w["us"] == 30.8 and abs(w["GBs"] - r["achieved"]) < 0.2
    assert abs(w["frac_of_8tbs"] - w["GBs"] / 8000) < 1e-4


def test_profile_traffic_follows_the_kernel_code(tmp_path, monkeypatch):
    """A committed ncu summary's traffic is used only while its code digest matches: a
    comment-only edit keeps it, a code edit drops it."""
    import shutil
    csrc = os.path.join(ROOT, "paged_kv_attention_09_gb300", "csrc")
    root = tmp_path / "r"
    shutil.copytree(csrc, root / "paged_kv_attention_09_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.code_digest("decode")
    (root / "profiles" / "decode_w.md").write_text(
        f"code_sha256: {digest}\ntraffic_bytes_per_launch: 1234\n")
    assert bench.traffic_from_profiles("decode", "w") == 1234.0
    src = root / "paged_kv_attention_09_gb300" / "csrc" / "decode.cu"
    src.write_text(src.read_text() + "\n// a comment\n/* and another */\n")
    assert bench.code_digest("decode") == digest
    assert bench.traffic_from_profiles("decode", "w") == 1234.0
    src.write_text(src.read_text() + "\nstatic int pkv_extra_symbol = 1;\n")
    assert bench.code_digest("decode") != digest
    assert bench.traffic_from_profiles("decode", "w") is None


def test_line_with_prefill_and_cpu_baselines(capsys, monkeypatch):
    """The mixed workload's line: prefill TFLOP/s against the measured BF16 peaks, and the
    oracle's all-core and single-core rates (the oracle itself replaced here)."""
    wl = W.workload("mixed")
    acc = bench.step_accounting(wl)
    kern = {k: {"ms": v, "replays": 5, "launches_per_graph": 50}
            for k, v in (("append", 0.006), ("decode", 0.0287), ("prefill", 0.0377))}
    monkeypatch.setattr(bench, "run_ours", lambda args, rank, world: dict(
        wl=wl, acc=acc, R=4, ms=0.08, kern=kern, clocks=None, e2e=None, fused=False,
        n_append=1028, workloads={}))
    monkeypatch.setattr(bench, "measured_hbm", lambda: (6794.5, "measured"))
    monkeypatch.setattr(bench, "measured_bf16", lambda: (1903.5, 1700.2, "measured"))
    calls = []

    def fake_rate(wl_, seconds, threads, fused=True, rope=False, oc=None, counts=None):
        calls.append(threads)
        return (0.5 if threads > 1 else 0.1), 1e6, "2/4 decode sequences", 1.0, [2, 1]
    monkeypatch.setattr(bench, "cpu_oracle_rate", fake_rate)
    import oracle
    monkeypatch.setattr(oracle, "cache_from_workload", lambda wl_: None)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "mixed", "--steps", "5",
                                      "--warmup", "3", "--no-e2e"])
    bench.main()
    d = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][-1])
    tf = acc["prefill_flops"] / 0.0377e-3 / 1e12
    assert abs(d["prefill"]["tflops"] - tf) < 0.1
    assert abs(d["prefill"]["frac_of_bf16_burst"] - tf / 1903.5) < 1e-3
    assert abs(d["prefill"]["frac_of_bf16_sustained"] - tf / 1700.2) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == 0.5 and cb["single_core"]["value"] == 0.1
    assert cb["cores"] == min(len(os.sched_getaffinity(0)), 2) and calls[-1] == 1


def test_kernel_graph_time_protocol():
    """A kernel's time is the median replay of a graph of 50 launches, over at least 5
    replays and at least 200 ms of timed replays."""
    replays = []

    def replay(g):
        replays.append(g)
        return 20.0 if len(replays) % 2 else 30.0  # ms per replay of 50 launches
    ms, n = bench.kernel_graph_ms(lambda k: ("graph", k), replay, 50)
    assert replays[0] == ("graph", 50)
    assert n == len(replays) - 1 >= 5            # one untimed warm replay first
    assert sum(20.0 if i % 2 else 30.0 for i in range(2, n + 2)) >= 200.0
    assert ms in (20.0 / 50, 30.0 / 50, 25.0 / 50)


def test_workload_entry_and_regression_compare():
    wl = W.workload("mixed")
    acc = bench.step_accounting(wl)
    kt = {"decode": {"ms": 0.028, "replays": 7, "launches_per_graph": 50},
          "prefill": {"ms": 0.040, "replays": 7, "launches_per_graph": 50}}
    e = bench.workload_entry(wl, acc, kt, 6652.7, (1935.2, 1754.5, "measured"))
    gbs = acc["decode"] / 28e-6 / 1e9
    assert abs(e["decode"]["GBs"] - gbs) < 0.1
    assert abs(e["decode"]["frac_of_measured"] - gbs / 6652.7) < 1e-4
    assert abs(e["decode"]["kv_tokens_per_s"] - 4 * 32768 / 28e-6) < 1.0
    tf = acc["prefill_flops"] / 40e-6 / 1e12
    assert abs(e["prefill"]["TFLOPs"] - tf) < 0.1
    assert abs(e["prefill"]["frac_of_bf16_burst"] - tf / 1935.2) < 1e-4
    prev = {"workloads": {"mixed": {"decode": {"us": 25.0}, "prefill": {"us": 40.0}}}}
    c = bench.compare_lines(prev, {"workloads": {"mixed": e}})
    assert c["regressions"] == ["mixed/decode"]          # 28 vs 25 us: 12% slower
    assert c["kernels"]["mixed/prefill"]["change"] == 0.0
