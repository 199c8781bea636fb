"""Benchmark: paged decode attention (append + decode [+ chunked prefill]) on GB300.

One step = one pass of the hot path over one batch: the new K/V rows go into the paged
cache and every batch of the workload runs (decode and, for the mixed workload, chunked
prefill): pkv_append of the new rows, then pkv_decode_attn / pkv_prefill_chunk_attn.
``--fused`` runs the decode batch as one fused launch instead (pkv_decode_step: append of
the new row and attention; the prefill chunks' rows still go through pkv_append), and
``--rope`` adds the rotary embedding of the new query and key at position context - 1 to
that launch.  The default workload is the batch-256 TinyLlama-shaped INT8
decode.  Inputs are synthetic and seeded; R replicas of every input rotate so that each
step reads data that is not in L2.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn achieved HBM GB/s & seq-tokens/s vs 8 TB/s roofline, 1 GB300"
ROPE_THETA = 10000.0
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED = 1900.0, 1700.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="tinyllama-int8")
    ap.add_argument("--replicas", type=int, default=0, help="0 = enough to exceed 4x L2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: oracle time over all warm-up and timed steps "
                         "(each step samples at least one sequence per batch)")
    ap.add_argument("--fused", action="store_true",
                    help="the decode batch as one pkv_decode_step launch")
    ap.add_argument("--rope", action="store_true",
                    help="with --fused: the step also applies the rotary embedding")
    ap.add_argument("--layers", type=int, default=1,
                    help="a step runs the hot path over this many layers (one cache each, "
                         "shared tables and lengths), as a model's decode step does")
    ap.add_argument("--graphs", action="store_true",
                    help="end-to-end leg: the step's launches through the bucketed "
                         "CUDA-graph executor (decode-only workloads)")
    ap.add_argument("--workloads", default="all",
                    help="comma-separated workloads whose kernels the line reports one by "
                         "one ('all': the five configurations and the FP8 / INT4 caches; "
                         "'none')")
    ap.add_argument("--profile", action="store_true",
                    help="a short run for a profiler: the warm-up and the K timed steps only "
                         "(no per-kernel table, no end-to-end leg, no CPU baseline); its "
                         "numbers are not benchmark values")
    ap.add_argument("--compare", default=None,
                    help="an earlier line of this benchmark (or a file holding one): report "
                         "every kernel's change and the ones more than 10%% slower")
    return ap.parse_args()


# ----------------------------------------------------------------------------- bytes

def esz(code):
    """Bytes per element of a source (new-row) dtype: float32 or bfloat16."""
    return {0: 4, 1: 2}[code]


def kv_token_bytes(wl):
    """Cache bytes of one token over all kv heads: its K and V rows, plus the two FP32
    scales of the coded formats (INT8, FP8 one byte per element; INT4 half a byte)."""
    D = wl.head_dim
    row = {0: 4 * D, 1: 2 * D, 2: D, 3: D, 4: D // 2}[wl.kv_dtype]
    return wl.num_kv_heads * (2 * row + (8 if wl.kv_dtype in (2, 3, 4) else 0))


def decode_bytes(wl, b):
    """Algorithmic HBM bytes of one decode call: every cached token's K and V (and the
    coded formats' scales) once, q, out, the used block-table entries and the lengths."""
    Hkv, D, Hq = wl.num_kv_heads, wl.head_dim, wl.num_q_heads
    per_tok = kv_token_bytes(wl)
    toks = int(b.context_lens.sum())
    pages = int(sum(math.ceil(int(L) / 16) for L in b.context_lens))
    qb = b.q.size * (2 if b.q.dtype == np.uint16 else 4)
    return toks * per_tok + qb + b.q.shape[0] * Hq * D * 4 + pages * 4 + b.num_seqs * 4


def prefill_bytes(wl, b):
    Hkv, D, Hq = wl.num_kv_heads, wl.head_dim, wl.num_q_heads
    per_tok = kv_token_bytes(wl)
    toks = int(b.context_lens.sum())
    pages = int(sum(math.ceil(int(L) / 16) for L in b.context_lens))
    qb = b.q.size * (2 if b.q.dtype == np.uint16 else 4)
    return toks * per_tok + qb + b.q.shape[0] * Hq * D * 4 + pages * 4 + (2 * b.num_seqs + 1) * 4


def prefill_flops(wl, b):
    f = 0
    for s in range(b.num_seqs):
        L, Lq = int(b.context_lens[s]), int(b.chunk_lens[s])
        keys = sum(L - Lq + i + 1 for i in range(Lq))
        f += 4 * keys * wl.head_dim * wl.num_q_heads
    return f


def append_bytes(wl):
    T = int(wl.step_rows.shape[0])
    Hkv, D = wl.num_kv_heads, wl.head_dim
    src = T * Hkv * D * esz(wl.new_dtype) * 2
    dst = T * kv_token_bytes(wl)
    return src + dst + T * 4


def step_accounting(wl):
    acc = {"append": append_bytes(wl), "decode": 0, "prefill": 0, "prefill_flops": 0,
           "kv_tokens": 0, "seqs": 0}
    for b in wl.batches:
        if b.kind == "decode":
            acc["decode"] += decode_bytes(wl, b)
            acc["kv_tokens"] += int(b.context_lens.sum())
            acc["seqs"] += b.num_seqs
        else:
            acc["prefill"] += prefill_bytes(wl, b)
            acc["prefill_flops"] += prefill_flops(wl, b)
    acc["total"] = acc["append"] + acc["decode"] + acc["prefill"]
    return acc


def workload_config(wl, layers=1):
    """The keys of the JSON line's config that identify the workload (both arms)."""
    return {"workload": wl.name, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "page_size": wl.page_size, "num_pages": wl.num_pages,
            "batches": [{"kind": b.kind, "num_seqs": b.num_seqs,
                         "context_tokens": int(b.context_lens.sum())} for b in wl.batches],
            "layers": layers}


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, device) -> float:
    """The largest value over the ranks of the default process group (the job's time is
    its slowest rank's); every rank gets it."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time
    (each rank runs the same workload: weak scaling)."""
    return units_per_rank * world / seconds


# ----------------------------------------------------------------------------- peaks, clocks

def measured_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16():
    """Measured dense BF16 TFLOP/s (burst, sustained) of the GB300s, or the
    fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r[1:])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": reasons}


def code_digest(kernel_tag):
    """sha256 of the code a kernel is built from: its .cu file and every header of the
    package's CUDA sources, with comments and blank space removed (a comment-only edit
    leaves the kernel, and so its profile, unchanged)."""
    csrc = os.path.join(ROOT, "paged_kv_attention_09_gb300", "csrc")
    names = [f"{kernel_tag}.cu"] + sorted(f for f in os.listdir(csrc) if f.endswith((".h", ".cuh")))
    h = hashlib.sha256()
    for name in names:
        text = open(os.path.join(csrc, name)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [" ".join(line.split()) for line in text.splitlines()]
        h.update(("\n".join(l for l in lines if l) + "\n").encode())
    return h.hexdigest()


def traffic_from_profiles(kernel_tag, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel code (its code digest is recorded in the summary)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    try:
        text = open(path).read()
        m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        s = re.search(r"code_sha256:\s*([0-9a-f]{64})", text)
        if m and s and s.group(1) == code_digest(kernel_tag):
            return float(m.group(1))
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- CPU oracle

def cpu_oracle_rate(wl, seconds, threads, fused=True, rope=False, oc=None, counts=None):
    """Time the oracle (as it stands) on a bounded sample of the workload: whole
    sequences of the decode batch (as the same fused step when ``fused``) and of the
    prefill batch, taken in order until about ``seconds`` of wall time (at least one
    sequence of each batch).  ``oc``: the oracle's cache of the workload, built here when
    not given (outside the timed calls).  ``counts``: run exactly that many sequences of
    each batch once, instead of searching for the sample size.  Returns (GB/s, tokens/s,
    sample description, timed seconds, sequences per batch)."""
    import oracle
    if oc is None:
        oc = oracle.cache_from_workload(wl)
    d0 = wl.batches[0]
    new_rows = wl.step_rows[:d0.num_seqs]
    done_bytes, done_tok, t_total, sample, used = 0, 0, 0.0, [], []
    for bi, b in enumerate(wl.batches):
        B = b.num_seqs
        # at least one sequence per host thread, so that every core the baseline reports works
        n = min(B, max(1, threads)) if counts is None else counts[bi]
        while True:
            seqs = list(range(min(B, n)))
            t0 = time.perf_counter()
            if b.kind == "decode" and fused:
                oracle.decode_step(oc, b.q, b.q_dtype, wl.k_src[new_rows], wl.v_src[new_rows],
                                   wl.new_dtype, wl.slots[new_rows],
                                   (b.context_lens - 1).astype(np.int32) if rope else None,
                                   ROPE_THETA,
                                   b.block_tables, b.context_lens, wl.scale, seqs=seqs,
                                   threads=threads)
            elif b.kind == "decode":
                oracle.decode(oc, b.q, b.q_dtype, b.block_tables, b.context_lens, wl.scale,
                              seqs=seqs, threads=threads)
            else:
                oracle.prefill(oc, b.q, b.q_dtype, b.q_start_loc, b.block_tables,
                               b.context_lens, wl.scale, seqs=seqs, threads=threads)
            dt = time.perf_counter() - t0
            if counts is not None or dt >= seconds / len(wl.batches) or len(seqs) == B:
                break
            n = max(n + 1, min(B, int(n * max(2.0, 0.8 * seconds / len(wl.batches) / max(dt, 1e-3)))))
        toks = int(sum(int(b.context_lens[s]) for s in seqs))
        per_tok = kv_token_bytes(wl)
        done_bytes += toks * per_tok
        done_tok += toks
        t_total += dt
        sample.append(f"{len(seqs)}/{B} {b.kind} sequences")
        used.append(len(seqs))
    return done_bytes / t_total / 1e9, done_tok / t_total, ", ".join(sample), t_total, used


# ----------------------------------------------------------------------------- GPU run

# Workloads whose kernels the line reports one by one: the five configurations of the
# benchmark (tiny, SmolLM2, Qwen2.5, TinyLlama INT8, mixed) and the FP8 / INT4 caches at
# the TinyLlama shapes.
ALL_WORKLOADS = ("tiny", "smollm2-f32", "qwen-bf16", "tinyllama-int8", "mixed",
                 "tinyllama-fp8", "tinyllama-int4")
KERNEL_LAUNCHES = 50      # launches per captured graph of one kernel
KERNEL_REPLAYS = 5        # at least this many timed replays of that graph ...
KERNEL_MIN_MS = 200.0     # ... and at least this much timed GPU time, for the clock record


def kernel_graph_ms(capture_fn, replay_fn, n_launch):
    """Time one kernel: a CUDA graph of ``n_launch`` launches (over rotating replicas),
    replayed at least KERNEL_REPLAYS times and until KERNEL_MIN_MS of timed region have
    passed; the median replay over ``n_launch`` is the time per launch.  Returns (ms per
    launch, replays)."""
    g = capture_fn(n_launch)
    replay_fn(g)  # warm
    times = []
    while len(times) < KERNEL_REPLAYS or (sum(times) < KERNEL_MIN_MS and len(times) < 20000):
        times.append(replay_fn(g))
    return statistics.median(times) / n_launch, len(times)


class Prepared:
    """A workload on the device: R replicas of every input (R x the step's bytes > 4x L2),
    each with `layers` caches, and the step's new rows."""

    def __init__(self, wl, dev, layers=1, replicas=0, fused=False, rope=False):
        import torch

        from paged_kv_attention_09_gb300 import runner
        self.wl, self.dev, self.NL = wl, dev, max(1, layers)
        self.acc = step_accounting(wl)  # per layer
        ws_bytes = self.acc["total"] * self.NL
        self.R = replicas or max(2, math.ceil(4 * L2_BYTES / max(ws_bytes, 1)))
        base = runner.upload(wl, f"cuda:{dev}")
        self.base = base
        self.fused = fused and wl.batches[0].kind == "decode"
        rows = base.step_rows
        self.dec_in = None
        if self.fused:  # the decode batch's new rows go through pkv_decode_step
            self.dec_in = runner.decode_step_inputs(base, 0, rope=rope)
            rows = rows[wl.batches[0].num_seqs:]
        self.step_k, self.step_v, self.step_s = (base.k_src[rows].contiguous(),
                                                 base.v_src[rows].contiguous(),
                                                 base.slots[rows].contiguous())
        self.n_append = int(self.step_s.numel())
        reps = [base]
        for _ in range(self.R - 1):
            batches = [runner.DeviceBatch(b.kind, b.q.clone(), b.block_tables.clone(),
                                          b.context_lens.clone(),
                                          None if b.q_start_loc is None else b.q_start_loc.clone(),
                                          b.max_q_len, torch.empty_like(b.out),
                                          None if b.workspace is None else torch.zeros_like(b.workspace))
                       for b in base.batches]
            reps.append(runner.DeviceWorkload(wl, base.cache.clone(), base.k_src, base.v_src,
                                              base.slots, base.step_rows, batches,
                                              base.dev_status))
        self.reps = reps
        # every replica's layers: the replica itself, then copies of its cache that share
        # its tables, lengths, queries and outputs
        self.layered = [[dw] + [runner.DeviceWorkload(wl, dw.cache.clone(), dw.k_src, dw.v_src,
                                                      dw.slots, dw.step_rows, dw.batches,
                                                      dw.dev_status)
                                for _ in range(self.NL - 1)] for dw in reps]
        self.stream = torch.cuda.Stream(device=f"cuda:{dev}")
        self.stream.wait_stream(torch.cuda.current_stream())
        self.names = (["append"] if self.n_append else []) + [b.kind for b in wl.batches]

    def run_j(self, dw, j, rope_theta=ROPE_THETA):
        from paged_kv_attention_09_gb300 import runner
        if self.fused and j == 0:
            runner.run_decode_step(dw, self.dec_in, 0, rope_theta, self.stream)
        else:
            runner.run_batch(dw, j, self.stream)

    def append_only(self, i):
        from paged_kv_attention_09_gb300 import pkv
        for dw in self.layered[i % self.R]:
            pkv.pkv_append(dw.cache, self.step_k, self.step_v, self.step_s, dw.dev_status,
                           self.stream)

    def batch_only(self, j):
        def run(i):
            for dw in self.layered[i % self.R]:
                self.run_j(dw, j)
        return run

    def step(self, i):
        from paged_kv_attention_09_gb300 import pkv
        for dw in self.layered[i % self.R]:
            if self.n_append:
                pkv.pkv_append(dw.cache, self.step_k, self.step_v, self.step_s, dw.dev_status,
                               self.stream)
            for j in range(len(self.wl.batches)):
                self.run_j(dw, j)

    def kernel_fns(self):
        """(name, launch function) of every kernel of the step, in order."""
        return ([("append", self.append_only)] if self.n_append else []) + \
            [(b.kind, self.batch_only(j)) for j, b in enumerate(self.wl.batches)]

    def capture(self, fn, k, first=0):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(k):
                fn(first + i)
        return g

    def replay_ms(self, g):
        # replay() launches on the current stream: make it the stream the events use
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def kernel_times(self):
        """Per-kernel time (ms per launch per layer) and replays, by kernel name."""
        out = {}
        for name, fn in self.kernel_fns():
            ms, reps = kernel_graph_ms(lambda n, fn=fn: self.capture(fn, n), self.replay_ms,
                                       KERNEL_LAUNCHES)
            out[name] = {"ms": ms / self.NL, "replays": reps, "launches_per_graph": KERNEL_LAUNCHES}
        return out

    def status(self):
        return int(self.base.dev_status.item())


def workload_entry(wl, acc, kt, peak, bf16):
    """The line's record of one workload's kernels: time per launch, and for the decode
    kernel its achieved GB/s against the measured copy peak and 8 TB/s, KV tokens/s and
    decode steps/s; for the prefill kernel TFLOP/s against the measured BF16 peaks."""
    burst, sustained, _ = bf16
    e = {}
    for name, t in kt.items():
        us = t["ms"] * 1e3
        rec = {"us": round(us, 3), "replays": t["replays"],
               "launches_per_graph": t["launches_per_graph"]}
        if name == "decode":
            gbs = acc["decode"] / (us * 1e-6) / 1e9
            rec.update({"GBs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                        "frac_of_8tbs": round(gbs / 8000.0, 4),
                        "kv_tokens_per_s": round(acc["kv_tokens"] / (us * 1e-6), 1),
                        "decode_steps_per_s": round(acc["seqs"] / (us * 1e-6), 1),
                        "bytes_per_launch": acc["decode"]})
        elif name == "prefill":
            tf = acc["prefill_flops"] / (us * 1e-6) / 1e12
            rec.update({"TFLOPs": round(tf, 1), "frac_of_bf16_burst": round(tf / burst, 4),
                        "frac_of_bf16_sustained": round(tf / sustained, 4),
                        "flops_per_launch": acc["prefill_flops"]})
        elif name == "append":
            rec["GBs"] = round(acc["append"] / (us * 1e-6) / 1e9, 1)
        e[name] = rec
    return e


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    from paged_kv_attention_09_gb300 import pkv
    from paged_kv_attention_09_gb300 import workloads as W

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    pkv.load()
    peak, _ = measured_hbm()
    bf16 = measured_bf16()
    wl = W.workload(args.workload)
    pr = Prepared(wl, dev, layers=args.layers, replicas=args.replicas, fused=args.fused,
                  rope=args.rope)
    acc, R, NL, K = pr.acc, pr.R, pr.NL, args.steps

    with torch.cuda.stream(pr.stream):
        for i in range(args.warmup):
            pr.step(i)
    torch.cuda.synchronize()
    if pr.status() != 0:
        raise RuntimeError(f"device status {pr.status()} after warm-up")

    # The K timed steps are one CUDA graph (launch overhead out of the timed region);
    # every kernel in it is ours.
    g_step = pr.capture(pr.step, K, args.warmup)
    with torch.cuda.stream(pr.stream):
        g_step.replay()
    torch.cuda.synchronize()
    wl_list = [] if args.workloads == "none" or args.profile else \
        (list(ALL_WORKLOADS) if args.workloads == "all" else args.workloads.split(","))
    tables = {}
    with ClockSampler(dev) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        total_ms = pr.replay_ms(g_step)
        if world > 1:
            dist.barrier()
        del g_step
        if args.profile:
            return {"wl": wl, "acc": acc, "R": R, "ms": total_ms / K, "kern": {},
                    "clocks": None, "e2e": None, "fused": pr.fused, "n_append": pr.n_append,
                    "workloads": {}}
        # per-kernel times: the benchmarked workload (its layers and step form), then every
        # other workload of the table, one at a time on the device
        kern = pr.kernel_times()
        tables[wl.name] = workload_entry(wl, acc, kern, peak, bf16)
        for name in wl_list:
            if name == wl.name:
                continue
            other = Prepared(W.workload(name), dev)
            with torch.cuda.stream(other.stream):
                for i in range(3):
                    other.step(i)
            torch.cuda.synchronize()
            if other.status() != 0:
                raise RuntimeError(f"device status {other.status()} on {name}")
            tables[name] = workload_entry(other.wl, other.acc, other.kernel_times(), peak, bf16)
            del other
            torch.cuda.empty_cache()
    if world > 1:
        total_ms = max_over_ranks(total_ms, f"cuda:{dev}")
    ms = total_ms / K

    # ---- end to end through the C ABI with host buffers: H2D of the step's inputs
    # (q, new K/V, slots, tables, lengths) from pinned memory, the calls, D2H of outputs
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, pr, world, dev, acc, K)
    if pr.status() != 0:
        raise RuntimeError(f"device status {pr.status()} after the timed steps")
    return {"wl": wl, "acc": acc, "R": R, "ms": ms, "kern": kern, "clocks": clk.summary(),
            "e2e": e2e, "fused": pr.fused, "n_append": pr.n_append, "workloads": tables}


class _Runtime:
    """The CUDA runtime's copy and event calls, issued through ctypes: the end-to-end loop
    orders its copies and launches with them at about a microsecond of host time each
    (a torch copy or event call costs several)."""

    def __init__(self):
        import ctypes
        import torch
        self.ct = ctypes
        self.rt = ctypes.CDLL(f"libcudart.so.{torch.version.cuda.split('.')[0]}")
        V, U = ctypes.c_void_p, ctypes.c_uint
        self.rt.cudaMemcpyAsync.argtypes = [V, V, ctypes.c_size_t, ctypes.c_int, V]
        self.rt.cudaEventRecord.argtypes = [V, V]
        self.rt.cudaStreamWaitEvent.argtypes = [V, V, U]
        self.rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(V), U]
        self.rt.cudaEventDestroy.argtypes = [V]
        self.events = []

    def event(self):
        e = self.ct.c_void_p()
        self.check(self.rt.cudaEventCreateWithFlags(self.ct.byref(e), 2), "event")  # no timing
        self.events.append(e)
        return e

    @staticmethod
    def check(code, what):
        if code != 0:
            raise RuntimeError(f"CUDA runtime error {code} ({what})")

    def close(self):
        for e in self.events:
            self.rt.cudaEventDestroy(e)
        self.events = []


def run_e2e(args, pr, world, dev, acc, K):
    """The same step through the public API with host buffers: every step copies its
    inputs from pinned host memory and its outputs back, inside the timed region."""
    import torch

    from paged_kv_attention_09_gb300 import pkv
    wl, NL, R, stream = pr.wl, pr.NL, pr.R, pr.stream
    step_dev = [pr.step_k, pr.step_v, pr.step_s] + \
        ([t for t in pr.dec_in if t is not None] if pr.fused else [])
    host_in = [t.cpu().pin_memory() for t in step_dev]
    for b in pr.base.batches:
        host_in += [b.q.cpu().pin_memory(), b.block_tables.cpu().pin_memory(),
                    b.context_lens.cpu().pin_memory()]
        if b.q_start_loc is not None:
            host_in.append(b.q_start_loc.cpu().pin_memory())
    host_out = [b.out.cpu().pin_memory() for b in pr.base.batches]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    graphs = None
    if args.graphs:
        if len(wl.batches) != 1 or wl.batches[0].kind != "decode":
            raise SystemExit("--graphs: decode-only workloads")
        gk, gv, gs, gp = pr.dec_in if pr.fused else (pr.step_k, pr.step_v, pr.step_s, None)
        graphs = []
        for dws in pr.layered:
            b = dws[0].batches[0]
            graphs.append(pkv.DecodeGraph(
                [pkv.GraphLayer(dw.cache, b.q, b.out, gk, gv) for dw in dws], b.block_tables,
                b.context_lens, wl.scale, [b.q.shape[0]], slot_mapping=gs, fused=pr.fused,
                positions=gp, rope_theta=ROPE_THETA, dev_status=dws[0].dev_status))

    def e2e_step(i):
        dw = pr.reps[i % R]
        dev_in = list(step_dev)
        for b in dw.batches:
            dev_in += [b.q, b.block_tables, b.context_lens]
            if b.q_start_loc is not None:
                dev_in.append(b.q_start_loc)
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)  # on `stream` (the current stream here)
        graphs[i % R].launch(dw.batches[0].q.shape[0], stream)
        for b, h in zip(dw.batches, host_out):
            h.copy_(b.out, non_blocking=True)

    # Direct launches: a step's inputs land on a copy stream while the previous step
    # computes, and its outputs are read back on another while the next one computes.
    # Every replica has its own copy of the step's new rows; events keep a replica's
    # inputs until its step has read them and its outputs until they are read back.
    from paged_kv_attention_09_gb300 import runner
    dec_r = [None if pr.dec_in is None else tuple(None if t is None else t.clone() for t in pr.dec_in)
             for _ in range(R)]
    step_r = [[pr.step_k.clone(), pr.step_v.clone(), pr.step_s.clone()] for _ in range(R)]
    h2d_s = torch.cuda.Stream(device=stream.device)
    d2h_s = torch.cuda.Stream(device=stream.device)
    used = [False] * R

    def dev_inputs(r):
        d = list(step_r[r]) + ([t for t in dec_r[r] if t is not None] if pr.fused else [])
        for b in pr.reps[r].batches:
            d += [b.q, b.block_tables, b.context_lens]
            if b.q_start_loc is not None:
                d.append(b.q_start_loc)
        return d

    # One copy per direction and step: every replica's inputs become views of one device
    # buffer (16-byte-aligned offsets) with the layout of one pinned host buffer.
    host_stage, dev_stage = None, []
    if graphs is None:
        torch.cuda.synchronize()
        sizes = [t.numel() * t.element_size() for t in host_in]
        offs, tot = [], 0
        for n in sizes:
            offs.append(tot)
            tot += (n + 15) // 16 * 16
        host_stage = torch.empty(tot, dtype=torch.uint8).pin_memory()
        for h, o, n in zip(host_in, offs, sizes):
            host_stage[o:o + n].copy_(h.reshape(-1).view(torch.uint8))
        for r in range(R):
            buf = torch.empty(tot, dtype=torch.uint8, device=stream.device)
            views = [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(dev_inputs(r), offs, sizes)]
            for v, t in zip(views, dev_inputs(r)):
                v.copy_(t)
            it = iter(views)
            step_r[r] = [next(it), next(it), next(it)]
            if pr.fused:
                dec_r[r] = tuple(None if t is None else next(it) for t in dec_r[r])
            for b in pr.reps[r].batches:
                b.q, b.block_tables, b.context_lens = next(it), next(it), next(it)
                if b.q_start_loc is not None:
                    b.q_start_loc = next(it)
            dev_stage.append(buf)

    # Per step: the input copy on h2d_s once the replica's previous step has read its
    # inputs, the step's launches on `stream` once the inputs have landed and the
    # replica's previous outputs were read back, then the output copy on d2h_s.  The
    # copies and events go straight to the CUDA runtime and the library calls are bound
    # once (pkv.BoundCall), so the host spends ~1 us per call instead of the ~45 us per
    # step that torch copies, events and the full wrappers cost.
    if graphs is None:
        import ctypes as ct
        rtm = _Runtime()
        rt = rtm.rt
        ev_in = [rtm.event() for _ in range(R)]
        ev_done = [rtm.event() for _ in range(R)]
        ev_out = [rtm.event() for _ in range(R)]
        cs = ct.c_void_p(stream.cuda_stream)
        hs = ct.c_void_p(h2d_s.cuda_stream)
        ds = ct.c_void_p(d2h_s.cuda_stream)
        nbytes = host_stage.numel()
        h2d_args, d2h_args, calls = [], [], []
        for r in range(R):
            h2d_args.append((ct.c_void_p(dev_stage[r].data_ptr()), ct.c_void_p(host_stage.data_ptr()),
                             nbytes, 1, hs))  # cudaMemcpyHostToDevice
            d2h_args.append([(ct.c_void_p(h.data_ptr()), ct.c_void_p(b.out.data_ptr()),
                              b.out.numel() * b.out.element_size(), 2, ds)  # DeviceToHost
                             for b, h in zip(pr.reps[r].batches, host_out)])
            sk, sv, ss = step_r[r]
            cr = []
            for dw in pr.layered[r]:
                if pr.n_append:
                    cr.append(pkv.pkv_append(dw.cache, sk, sv, ss, dw.dev_status, stream, bound=True))
                for j in range(len(wl.batches)):
                    if pr.fused and j == 0:
                        cr.append(runner.run_decode_step(dw, dec_r[r], 0, ROPE_THETA, stream, bound=True))
                    else:
                        cr.append(runner.run_batch(dw, j, stream, bound=True))
            calls.append(cr)
        memcpy, record, wait, check = rt.cudaMemcpyAsync, rt.cudaEventRecord, rt.cudaStreamWaitEvent, rtm.check

    def piped_step(i):
        r = i % R
        if used[r]:
            check(wait(hs, ev_done[r], 0), "wait")  # the replica's previous step read its inputs
        check(memcpy(*h2d_args[r]), "input copy")
        check(record(ev_in[r], hs), "record")
        check(wait(cs, ev_in[r], 0), "wait")
        if used[r]:
            check(wait(cs, ev_out[r], 0), "wait")  # its previous outputs were read back
        for c in calls[r]:
            c()
        check(record(ev_done[r], cs), "record")
        check(wait(ds, ev_done[r], 0), "wait")
        for a in d2h_args[r]:
            check(memcpy(*a), "output copy")
        check(record(ev_out[r], ds), "record")
        used[r] = True

    run = e2e_step if graphs is not None else piped_step
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            run(i)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        h2d_s.wait_event(s2)
        d2h_s.wait_event(s2)
        for i in range(K):
            run(i)
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)
        e2.record(stream)
        torch.cuda.synchronize()
    e2e_ms = s2.elapsed_time(e2) / K
    if world > 1:
        e2e_ms = max_over_ranks(e2e_ms, f"cuda:{dev}")
    if graphs is not None:
        for g in graphs:
            g.close()
    else:
        rtm.close()
    return {"value": round(job_rate(acc["total"] * NL, world, e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 5),
            "launches": "one CUDA graph per step" if graphs is not None
            else "direct; a step's input copies and the previous step's output copy overlap its "
                 "kernels; copies and events through the CUDA runtime, library calls bound once"}


def compare_lines(prev, line, threshold=0.10):
    """Per-kernel regression check against an earlier line of this benchmark: every
    kernel time of the `workloads` table present in both, its relative change, and the
    kernels slower by more than `threshold`."""
    out, slow = {}, []
    for wname, kernels in line.get("workloads", {}).items():
        for kname, rec in kernels.items():
            old = prev.get("workloads", {}).get(wname, {}).get(kname)
            if not old or not old.get("us") or "us" not in rec:
                continue
            ch = rec["us"] / old["us"] - 1.0
            key = f"{wname}/{kname}"
            out[key] = {"prev_us": old["us"], "us": rec["us"], "change": round(ch, 4)}
            if ch > threshold:
                slow.append(key)
    return {"threshold": threshold, "kernels": out, "regressions": slow}


def read_line(path):
    """The last JSON object line of a file (a bench line, or a driver record holding one
    under parsed / in its output)."""
    text = open(path).read()
    try:
        d = json.loads(text)
        if isinstance(d, dict):
            if "workloads" in d:
                return d
            for k in ("parsed",):
                if isinstance(d.get(k), dict):
                    return d[k]
            text = json.dumps(d)
    except ValueError:
        pass
    found = None
    for m in re.finditer(r'\{"metric".*?\}(?=\s*(?:\\n|\n|$))', text):
        try:
            found = json.loads(m.group(0).encode().decode("unicode_escape"))
        except ValueError:
            continue
    if found is None:
        raise ValueError(f"no bench line in {path}")
    return found


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank != 0:
            return
        return main_reference(args)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_ours(args, rank, world)
    wl, acc, R, ms, kern = r["wl"], r["acc"], r["R"], r["ms"], r["kern"]
    clocks, e2e, fused, n_append = r["clocks"], r["e2e"], r["fused"], r["n_append"]
    K = args.steps
    avg = {n: v["ms"] for n, v in kern.items()}
    from paged_kv_attention_09_gb300 import workloads as W
    peak, peak_kind = measured_hbm()
    NL = max(1, args.layers)
    value = job_rate(acc["total"] * NL, world, ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[wl.kv_dtype] + "-kv/f32-acc",
        "data": "synthetic (seeded N(0,1) values, shapes of the named model family)",
        "config": {
            **workload_config(wl, NL),
            "step": ((("decode batch as one fused launch (rotary embedding of the new query and "
                       "key, append of the new row, attention)") if args.rope else
                      "decode batch as one fused launch (append of the new row, attention)") +
                     ("; prefill chunk rows appended, then prefill attention"
                      if len(wl.batches) > 1 else "") if fused else
                     "append new K/V rows, then attention over every batch"),
            "timing": ("value: CUDA events around one CUDA-graph replay of the K steps; "
                       f"kernels: median of >= {KERNEL_REPLAYS} replays of a graph of "
                       f"{KERNEL_LAUNCHES} launches, replayed for >= {KERNEL_MIN_MS:.0f} ms"),
            "bytes_per_step": acc["total"] * NL, "replicas": R,
            "l2": f"rotating {R} replicas of every input ({R} x {acc['total'] * NL / 1e6:.1f} MB "
                  f"per cycle > {L2_BYTES / 2**20:.0f} MiB L2)",
            "parallelism": "replicas" if world > 1 else "single",
        },
        "seq_tokens_per_s": round(acc["kv_tokens"] * NL * world / (ms * 1e-3), 1),
        "decode_steps_per_s": round(acc["seqs"] * world / (ms * 1e-3), 1),
        "kernel_ms": {n: round(v, 5) for n, v in avg.items()},
        "gpu_launches": K * NL * ((1 if n_append else 0) + len(wl.batches)),
    }
    dec = avg.get("decode")
    if dec:
        achieved = acc["decode"] / (dec * 1e-3) / 1e9
        line["roofline"] = {"bound": "hbm",
                            "kernel": "decode_kernel (fused step)" if fused else "decode_kernel",
                            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                            "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                            "frac_of_8tbs": round(achieved / 8000.0, 4),
                            "traffic": traffic_from_profiles("decode", wl.name),
                            "algorithmic_bytes_per_launch": acc["decode"]}
    if "prefill" in avg:
        tf = acc["prefill_flops"] / (avg["prefill"] * 1e-3) / 1e12
        burst, sustained, src = measured_bf16()
        line["prefill"] = {"ms": round(avg["prefill"], 5), "tflops": round(tf, 1),
                           "frac_of_bf16_burst": round(tf / burst, 4),
                           "frac_of_bf16_sustained": round(tf / sustained, 4),
                           "peak_source": src}
    if r.get("workloads"):
        line["workloads"] = r["workloads"]
    if e2e:
        line["e2e"] = e2e
    line["clocks"] = clocks
    if args.compare:
        line["compare"] = compare_lines(read_line(args.compare), line)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        threads = len(os.sched_getaffinity(0))
        import oracle
        oc = oracle.cache_from_workload(wl)  # built once for both samples
        gbs, tps, sample, secs, used = cpu_oracle_rate(wl, args.cpu_sample_seconds, threads, fused,
                                                       args.rope, oc)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s",
                                "cores": min(threads, max(used)),
                                "kind": "oracle", "sample": sample + f" ({secs:.1f} s wall)",
                                "seq_tokens_per_s": round(tps, 1)}
        # the same oracle on one core, on a shorter sample
        gbs1, tps1, sample1, secs1, _ = cpu_oracle_rate(wl, args.cpu_sample_seconds / 4, 1,
                                                        fused, args.rope, oc)
        line["cpu_baseline"]["single_core"] = {
            "value": round(gbs1, 4), "unit": "GB/s", "seq_tokens_per_s": round(tps1, 1),
            "sample": sample1 + f" ({secs1:.1f} s wall)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_reference(args):
    """The oracle as it stands, on the host cores, one bounded sample per step."""
    import oracle
    from paged_kv_attention_09_gb300 import workloads as W
    wl = W.workload(args.workload)
    threads = len(os.sched_getaffinity(0))
    oc = oracle.cache_from_workload(wl)  # once, outside every step
    # the first warm-up step finds the sample size (sequences per batch) that takes about
    # the per-step share of the budget; every later step runs exactly that sample once
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    counts = None
    for _ in range(max(1, args.warmup)):
        *_, took, used = cpu_oracle_rate(wl, per_step, threads, args.fused, args.rope, oc, counts)
        if counts is None:
            # a sample of one sequence per core that overruns its share of the budget
            # falls back to one sequence (on one core) per batch
            counts = [1] * len(used) if took > 2 * per_step else used
    vals, secs = [], 0.0
    for _ in range(args.steps):
        gbs, tps, sample, s, _ = cpu_oracle_rate(wl, per_step, threads, args.fused, args.rope,
                                                 oc, counts)
        vals.append(gbs)
        secs += s
    v = statistics.fmean(vals)
    line = {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "impl": "reference",
            "dtype": "f64",
            "data": "synthetic (seeded N(0,1) values, shapes of the named model family)",
            "config": {**workload_config(wl, max(1, args.layers)),
                       "timing": "host wall clock around the oracle's bounded sample"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s",
                             "cores": min(threads, max(counts)),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
