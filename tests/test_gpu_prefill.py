"""Chunked-prefill attention on the GPU vs the FP64 oracle (BF16 KV cache).

Chunks of assorted lengths (1 token, page-aligned, ragged, longer than a tile) over
assorted prior contexts (none, partial page, several tiles); FP32 and BF16 queries;
NaN-poisoned padding; device-side errors; sampled rows of the full-size mixed workload.
"""
import os

import numpy as np
import pytest

import oracle
from paged_kv_attention_09_gb300 import pkv
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import gpu_outputs, max_err, oracle_outputs

pytestmark = pytest.mark.gpu

CHUNKS = [(0, 1), (0, 16), (5, 1), (20, 13), (16, 48), (33, 70), (130, 65), (0, 150)]


@pytest.mark.parametrize("Hq,Hkv,D,qd", [(12, 2, 128, W.BF16), (12, 2, 128, W.F32),
                                         (8, 8, 64, W.BF16), (4, 1, 64, W.F32),
                                         (16, 2, 128, W.BF16)])
def test_prefill_small_parity(Hq, Hkv, D, qd):
    wl = W.small_workload(3000 + Hq + D + qd, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          kv_dtype=W.BF16, q_dtype=qd, prefill=CHUNKS)
    ref = oracle_outputs(wl)[0]
    got, status, _ = gpu_outputs(wl)
    assert status == 0
    assert max_err(got[0], ref) <= 2e-3


def test_prefill_poisoned_padding():
    wl = W.small_workload(3100, num_q_heads=6, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(3, 9), (40, 21)], max_prefill_len=128)
    ref = oracle_outputs(wl)[0]
    got, status, _ = gpu_outputs(wl, cache_fill=float("nan"))
    assert status == 0
    assert np.all(np.isfinite(got[0]))
    assert max_err(got[0], ref) <= 2e-3


def test_prefill_bad_inputs_give_nan_rows_and_status():
    wl = W.small_workload(3101, num_q_heads=4, num_kv_heads=2, head_dim=64, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(10, 10), (10, 10), (10, 10)],
                          max_prefill_len=64)
    b = wl.batches[0]
    b.block_tables[0, 1] = -5                  # bad page
    b.context_lens[1] = 5                      # chunk (10) longer than the context
    got, status, _ = gpu_outputs(wl)
    assert status & pkv.DEV_BAD_PAGE and status & pkv.DEV_BAD_CHUNK
    assert np.all(np.isnan(got[0][0:10])) and np.all(np.isnan(got[0][10:20]))
    assert np.all(np.isfinite(got[0][20:30]))


# Long chunks over long contexts so that every split has several key tiles, plus a short
# chunk (one row tile) whose last split gets few or no key tiles.
SPLIT_CHUNKS = [(700, 300), (1500, 64), (0, 260), (30, 5)]


@pytest.mark.parametrize("Hq,Hkv,D,qd", [(12, 2, 128, W.BF16), (8, 2, 64, W.F32)])
def test_prefill_every_key_split(Hq, Hkv, D, qd):
    """Each key split (1, 2, 3 blocks per row tile, merged through the workspace by the
    last of them) within tolerance of the oracle, and equal to the unsplit result up to
    float rounding."""
    wl = W.small_workload(3200 + D, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          kv_dtype=W.BF16, q_dtype=qd, prefill=SPLIT_CHUNKS)
    ref = oracle_outputs(wl)[0]
    got = {}
    for key_split in (1, 2, 3):
        out, status, dw = gpu_outputs(wl, key_split=key_split)
        assert status == 0
        assert (dw.batches[0].workspace is None) == (key_split == 1)
        assert np.all(np.isfinite(out[0]))
        assert max_err(out[0], ref) <= 2e-3, key_split
        got[key_split] = out[0]
    assert max_err(got[2], got[1]) <= 1e-5 and max_err(got[3], got[1]) <= 1e-5


def test_prefill_split_bad_inputs_give_nan_rows():
    """A device-side error in a split row tile turns exactly its sequence's rows into NaN,
    through the merge too."""
    wl = W.small_workload(3210, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(600, 40), (600, 40), (600, 40)])
    b = wl.batches[0]
    b.block_tables[0, 30] = -5                 # bad page inside the first sequence's range
    b.context_lens[1] = 5                      # chunk (40) longer than the context
    got, status, _ = gpu_outputs(wl, key_split=3)
    assert status & pkv.DEV_BAD_PAGE and status & pkv.DEV_BAD_CHUNK
    assert np.all(np.isnan(got[0][0:80]))
    ref = oracle_outputs(wl, seqs=[2])[0]
    assert max_err(got[0][80:120], ref[80:120]) <= 2e-3


def test_prefill_lq1_matches_decode():
    """A one-token chunk is a decode step: both kernels must agree within tolerance."""
    wl = W.small_workload(3102, num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(77, 1), (0, 1), (300, 1)])
    got_p, _, _ = gpu_outputs(wl)
    b = wl.batches[0]
    dec = W.Batch("decode", b.context_lens, b.block_tables, b.q, b.q_dtype)
    wl.batches = [dec]
    got_d, _, _ = gpu_outputs(wl)
    assert max_err(got_p[0], got_d[0]) <= 2e-3


def _oracle_prefill_by_pieces(oc, b, scale, pieces):
    """The oracle's prefill of batch b, computed as `pieces` row ranges per sequence on a
    thread pool: rows r0..r1-1 of a chunk of Lq rows over context L are themselves a
    causal chunk of r1 - r0 rows over context L - (Lq - r1) (each row keeps its position
    and sees the same keys), so the pieces together are the whole chunk."""
    from concurrent.futures import ThreadPoolExecutor
    jobs = []
    for s in range(b.num_seqs):
        q0, q1 = int(b.q_start_loc[s]), int(b.q_start_loc[s + 1])
        Lq, L = q1 - q0, int(b.context_lens[s])
        cuts = np.linspace(0, Lq, pieces + 1).astype(int)
        for r0, r1 in zip(cuts[:-1], cuts[1:]):
            if r1 > r0:
                jobs.append((s, q0 + r0, q0 + r1, L - (Lq - r1)))
    out = np.full(b.q.shape, np.nan)

    def run(job):
        s, a0, a1, ctx = job
        out[a0:a1] = oracle.prefill(oc, b.q[a0:a1], b.q_dtype,
                                    np.array([0, a1 - a0], np.int32),
                                    b.block_tables[s:s + 1], np.array([ctx], np.int32), scale)
    with ThreadPoolExecutor(max(1, len(os.sched_getaffinity(0)))) as ex:
        list(ex.map(run, jobs))
    return out


def test_mixed_full_size_prefill_every_row():
    """The mixed workload's two 512-token chunks over 2048 prior tokens, in the
    benchmark's launch configuration: every (chunk row, head) against the oracle."""
    wl = W.workload("mixed")
    got, status, _ = gpu_outputs(wl)
    assert status == 0
    i = [k for k, b in enumerate(wl.batches) if b.kind == "prefill"][0]
    b = wl.batches[i]
    oc = oracle.cache_from_workload(wl)
    ref = _oracle_prefill_by_pieces(oc, b, wl.scale, pieces=8)
    assert got[i].shape == ref.shape == (1024, 12, 128)
    assert max_err(got[i], ref) <= 2e-3
    assert np.all(np.isfinite(got[i]))
