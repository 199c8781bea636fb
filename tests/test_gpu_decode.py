"""Decode attention on the GPU vs the FP64 oracle.

Element-by-element parity on small workloads spanning several pages, ragged tails,
every dtype combination and head layout; sampled parity at the full workload sizes in
the benchmark's launch configuration; NaN-poisoned padding; page-permutation
bit-identity; split-count invariance and determinism; device-side error reporting.
Tolerances (max abs error): 1e-4 for FP32 KV, 2e-3 for BF16 / INT8 / FP8 / INT4 KV.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import TOL, gpu_outputs, max_err, oracle_outputs

pytestmark = pytest.mark.gpu

LENS = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257]
SMALL = [
    # kv, q, Hq, Hkv, D
    (W.F32, W.F32, 9, 3, 64),
    (W.F32, W.BF16, 8, 2, 64),
    (W.F32, W.F32, 8, 2, 128),
    (W.F32, W.F32, 12, 1, 64),     # 12 heads -> two head groups
    (W.BF16, W.BF16, 12, 2, 128),
    (W.BF16, W.F32, 12, 2, 128),
    (W.BF16, W.BF16, 8, 8, 64),    # MHA
    (W.BF16, W.BF16, 16, 1, 128),  # MQA, two head groups
    (W.INT8, W.F32, 32, 4, 64),
    (W.INT8, W.BF16, 6, 2, 128),
    (W.INT8, W.F32, 4, 4, 64),
    (W.FP8, W.F32, 32, 4, 64),
    (W.FP8, W.BF16, 6, 2, 128),
    (W.FP8, W.F32, 12, 1, 64),     # two head groups
    (W.INT4, W.F32, 32, 4, 64),
    (W.INT4, W.BF16, 6, 2, 128),
    (W.INT4, W.F32, 12, 1, 128),   # two head groups
]


@pytest.mark.parametrize("kv,qd,Hq,Hkv,D", SMALL)
def test_decode_small_parity(kv, qd, Hq, Hkv, D):
    wl = W.small_workload(1000 + Hq * 10 + D + kv, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          kv_dtype=kv, q_dtype=qd, decode_lens=LENS)
    ref = oracle_outputs(wl)[0]
    got, status, _ = gpu_outputs(wl)
    assert status == 0
    assert max_err(got[0], ref) <= TOL[kv]


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_decode_poisoned_padding_is_never_read(kv):
    """Unwritten slots hold NaN (NaN scales for the coded formats, and NaN codes for FP8);
    table entries past the context
    hold -1.  Any read of either would show up as NaN or a bad-page status."""
    wl = W.small_workload(77 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[1, 17, 30, 47], max_decode_len=80)
    ref = oracle_outputs(wl)[0]
    got, status, _ = gpu_outputs(wl, cache_fill=float("nan"))
    assert status == 0
    assert np.all(np.isfinite(got[0]))
    assert max_err(got[0], ref) <= TOL[kv]


def test_decode_zero_length_gives_zero_rows():
    wl = W.small_workload(90, num_q_heads=6, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, decode_lens=[0, 5, 0], max_decode_len=32)
    got, status, _ = gpu_outputs(wl)
    assert status == 0
    assert np.all(got[0][0] == 0) and np.all(got[0][2] == 0)
    assert max_err(got[0], oracle_outputs(wl)[0]) <= 2e-3


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_page_permutation_bit_identical(kv):
    wl = W.small_workload(91 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[70, 33, 129])
    got1, _, _ = gpu_outputs(wl, chunk_pages=3)
    rng = np.random.default_rng(5)
    sigma = rng.permutation(wl.num_pages).astype(np.int32)
    b = wl.batches[0]
    b.block_tables = np.where(b.block_tables >= 0, sigma[np.maximum(b.block_tables, 0)], -1)
    wl.slots = (sigma[wl.slots // 16] * 16 + wl.slots % 16).astype(np.int32)
    got2, _, _ = gpu_outputs(wl, chunk_pages=3)
    assert np.array_equal(got1[0], got2[0])


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_split_count_invariance_and_determinism(kv):
    wl = W.small_workload(95 + kv, num_q_heads=12, num_kv_heads=2, head_dim=128 if kv else 64,
                          kv_dtype=kv, q_dtype=W.BF16 if kv == W.BF16 else W.F32,
                          decode_lens=[300, 1, 45, 160])
    ref = oracle_outputs(wl)[0]
    for chunk in (1, 2, 3, 5, 8, 19, 0):
        got, status, _ = gpu_outputs(wl, chunk_pages=chunk)
        again, _, _ = gpu_outputs(wl, chunk_pages=chunk)
        assert status == 0
        assert np.array_equal(got[0], again[0]), f"chunk {chunk} not deterministic"
        assert max_err(got[0], ref) <= TOL[kv], f"chunk {chunk}"


def test_bad_page_and_bad_length_give_nan_rows_and_status():
    wl = W.small_workload(97, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=W.BF16,
                          q_dtype=W.BF16, decode_lens=[40, 40, 40], max_decode_len=64)
    b = wl.batches[0]
    b.block_tables[1, 2] = wl.num_pages + 3       # bad page in sequence 1
    b.context_lens[2] = b.max_blocks * 16 + 1     # bad length in sequence 2
    for chunk in (0, 1):
        got, status, _ = gpu_outputs(wl, chunk_pages=chunk)
        assert status == pkv.DEV_BAD_PAGE | pkv.DEV_BAD_LEN
        assert np.all(np.isnan(got[0][1])) and np.all(np.isnan(got[0][2]))
        assert np.all(np.isfinite(got[0][0]))


def test_workspace_is_left_zero_for_the_next_call():
    wl = W.small_workload(98, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=W.INT8,
                          q_dtype=W.F32, decode_lens=[200, 200])
    dw = runner.upload(wl, split_pages=1)  # 13 splits: merged through the workspace
    ws = dw.batches[0].workspace
    assert ws is not None
    first = None
    for _ in range(3):
        runner.run_batch(dw, 0)
        torch.cuda.synchronize()
        o = dw.batches[0].out.cpu().numpy()
        first = o if first is None else first
        assert np.array_equal(o, first)
    tickets = ws[: 2 * 2].cpu().numpy()  # B * Hkv tickets lead the workspace
    assert not tickets.any()


# Full-size workloads in the benchmark's launch configuration (automatic split); the
# oracle computes every sequence, threaded over the host cores.
FULL = ["tiny", "smollm2-f32", "qwen-bf16", "tinyllama-int8", "mixed", "tinyllama-fp8",
        "tinyllama-int4"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity_every_row(name):
    wl = W.workload(name)
    got, status, _ = gpu_outputs(wl)
    assert status == 0
    oc = oracle.cache_from_workload(wl)
    i = [k for k, b in enumerate(wl.batches) if b.kind == "decode"][0]
    b = wl.batches[i]
    ref = oracle.decode(oc, b.q, b.q_dtype, b.block_tables, b.context_lens, wl.scale,
                        threads=len(os.sched_getaffinity(0)))
    assert got[i].shape == ref.shape
    assert max_err(got[i], ref) <= TOL[wl.kv_dtype]
    assert np.all(np.isfinite(got[i]))


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
@pytest.mark.parametrize("chunk", [0, 1000])
def test_long_context_many_iterations_per_warp(kv, chunk):
    """A single block streaming ~300 pages gives each warp more than two batches of 32
    iterations (the page-id prefetch rolls over); chunk 0 is the automatic split."""
    wl = W.small_workload(99 + kv, num_q_heads=8, num_kv_heads=1, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[16 * 300 - 5, 16 * 97 + 3])
    ref = oracle_outputs(wl)[0]
    got, status, _ = gpu_outputs(wl, chunk_pages=chunk)
    assert status == 0
    assert max_err(got[0], ref) <= TOL[kv]
