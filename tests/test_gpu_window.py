"""Sliding-window attention on the GPU ("tinyloop Current Status", KV cache modes table: a
cache window bounds the KV storage) vs the FP64 oracle: decode, chunked prefill and the
fused decode step, with windows shorter than a page, page-aligned, ragged and longer than
the context; splits that cut the window; released pages before the window (-1 table
entries); stale NaN rows before the window inside its first page."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import TOL, cache_bytes_equal, max_err

pytestmark = pytest.mark.gpu

DECODE_LENS = [45, 16, 1, 70, 300, 17, 129]


def decode_gpu(wl, window, bt=None, chunk=0, poison_rows=None):
    """Upload the workload (optionally NaN source rows at `poison_rows`), run windowed
    decode with table `bt`; returns (output, status, device workload)."""
    if poison_rows is not None:
        wl.k_src = wl.k_src.copy()
        wl.v_src = wl.v_src.copy()
        nan = np.uint16(0x7FC0) if wl.new_dtype == W.BF16 else np.float32("nan")
        wl.k_src[poison_rows] = nan
        wl.v_src[poison_rows] = nan
    dw = runner.upload(wl, "cuda", fill_history=False, split_pages=chunk)
    dw.cache.window = window
    runner.append_rows(dw, torch.arange(wl.slots.shape[0], device="cuda"))
    b = dw.batches[0]
    if bt is not None:
        b.block_tables.copy_(torch.from_numpy(bt))
    ws = pkv.pkv_decode_workspace_size(dw.cache, b.q.shape[0], wl.num_q_heads,
                                       wl.batches[0].max_blocks, chunk)
    b.workspace = pkv.workspace_for(ws, "cuda")
    runner.run_batch(dw, 0)
    torch.cuda.synchronize()
    return b.out.cpu().numpy().astype(np.float64), int(dw.dev_status.item()), dw


@pytest.mark.parametrize("kv,qd,Hq,Hkv,D", [(W.F32, W.F32, 9, 3, 64), (W.F32, W.BF16, 8, 2, 128),
                                            (W.BF16, W.BF16, 12, 2, 128), (W.BF16, W.F32, 8, 8, 64),
                                            (W.INT8, W.F32, 32, 4, 64), (W.INT8, W.BF16, 6, 1, 128),
                                            (W.FP8, W.F32, 8, 2, 64), (W.INT4, W.F32, 8, 2, 128)])
@pytest.mark.parametrize("window", [1, 5, 16, 17, 100, 1000])
def test_window_decode_matches_oracle(kv, qd, Hq, Hkv, D, window):
    wl = W.small_workload(8000 + kv * 10 + D + qd, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          kv_dtype=kv, q_dtype=qd, decode_lens=DECODE_LENS)
    b = wl.batches[0]
    ref = oracle.decode(oracle.cache_from_workload(wl), b.q, qd, b.block_tables, b.context_lens,
                        wl.scale, window=window)
    for chunk in (0, 2):  # automatic split, and a forced split that cuts the window
        got, status, _ = decode_gpu(wl, window, chunk=chunk)
        assert status == 0
        assert max_err(got, ref) <= TOL[kv], (chunk, max_err(got, ref))


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_window_released_pages_and_stale_nan_rows(kv):
    """Pages wholly before the window hold -1 in the table; the rows before the window in
    its first page are NaN: neither is read into the result."""
    window = 37
    lens = [200, 100, 38, 37, 36, 300]
    wl = W.small_workload(8100 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=lens)
    b = wl.batches[0]
    ref = oracle.decode(oracle.cache_from_workload(wl), b.q, W.F32, b.block_tables,
                        b.context_lens, wl.scale, window=window)
    bt = b.block_tables.copy()
    poison, row = [], 0
    for s, L in enumerate(lens):
        lo = max(0, L - window)
        bt[s, :lo // 16] = -1
        poison.extend(range(row + (lo // 16) * 16, row + lo))  # same page as the window start
        row += L
    plain, st0, _ = decode_gpu(wl, window)
    got, status, _ = decode_gpu(wl, window, bt=bt, poison_rows=np.array(poison, np.int64))
    assert st0 == 0 and status == 0
    assert np.all(np.isfinite(got))
    assert max_err(got, ref) <= TOL[kv]
    assert np.array_equal(got, plain)  # the same pages in the same order: bit-identical


def test_window_workspace_not_larger():
    """A window bounds the pages a sequence spans, so the split scratch can only shrink."""
    c = pkv.KVCache.allocate(8, 4, 64, W.INT8, "cuda")
    full = pkv.pkv_decode_workspace_size(c, 4, 32, 1024)
    c.window = 256
    assert 0 < full and pkv.pkv_decode_workspace_size(c, 4, 32, 1024) <= full


PREFILL_CHUNKS = [(0, 1), (0, 16), (5, 1), (20, 13), (16, 48), (33, 70), (130, 65), (0, 150),
                  (300, 40)]


@pytest.mark.parametrize("Hq,Hkv,D,qd", [(12, 2, 128, W.BF16), (12, 2, 128, W.F32),
                                         (8, 8, 64, W.BF16), (4, 1, 64, W.F32)])
@pytest.mark.parametrize("window", [1, 16, 50, 100, 1000])
def test_window_prefill_matches_oracle(Hq, Hkv, D, qd, window):
    wl = W.small_workload(8300 + Hq + D + qd, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          kv_dtype=W.BF16, q_dtype=qd, prefill=PREFILL_CHUNKS)
    b = wl.batches[0]
    ref = oracle.prefill(oracle.cache_from_workload(wl), b.q, qd, b.q_start_loc, b.block_tables,
                         b.context_lens, wl.scale, window=window)
    dw = runner.upload(wl, "cuda")
    dw.cache.window = window
    runner.append_rows(dw, dw.step_rows)
    runner.run_batch(dw, 0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    assert max_err(got, ref) <= 2e-3


def test_window_prefill_released_pages():
    """Prefill rows never read pages wholly before the lowest window start of the chunk."""
    window = 40
    wl = W.small_workload(8400, num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(200, 30), (90, 64), (10, 20)])
    b = wl.batches[0]
    ref = oracle.prefill(oracle.cache_from_workload(wl), b.q, W.BF16, b.q_start_loc,
                         b.block_tables, b.context_lens, wl.scale, window=window)
    bt = b.block_tables.copy()
    for s in range(b.num_seqs):
        first = int(b.context_lens[s]) - int(b.chunk_lens[s])  # the chunk's first position
        bt[s, :max(0, first - window + 1) // 16] = -1
    dw = runner.upload(wl, "cuda")
    dw.cache.window = window
    runner.append_rows(dw, dw.step_rows)
    dw.batches[0].block_tables.copy_(torch.from_numpy(bt))
    runner.run_batch(dw, 0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    assert max_err(got, ref) <= 2e-3


@pytest.mark.parametrize("kv,nd", [(W.F32, W.F32), (W.BF16, W.BF16), (W.INT8, W.F32)])
@pytest.mark.parametrize("window", [1, 20, 64])
def test_window_fused_step(kv, nd, window):
    wl = W.small_workload(8500 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, new_dtype=nd, decode_lens=[100, 16, 1, 65, 300])
    b = wl.batches[0]
    rows = wl.step_rows[:b.num_seqs]
    slots = wl.slots[rows].astype(np.int32)
    pos = (b.context_lens - 1).astype(np.int32)
    oc = oracle.cache_from_workload(wl, rows=wl.history_rows)
    ref = oracle.decode_step(oc, b.q, W.F32, wl.k_src[rows], wl.v_src[rows], nd, slots, pos,
                             1.0e4, b.block_tables, b.context_lens, wl.scale, window=window)
    for chunk in (0, 3):
        dw = runner.upload(wl, "cuda", split_pages=chunk)
        dw.cache.window = window
        inp = runner.decode_step_inputs(dw, 0, True)
        runner.run_decode_step(dw, inp, 0, 1.0e4)
        torch.cuda.synchronize()
        assert int(dw.dev_status.item()) == 0
        got = dw.batches[0].out.cpu().numpy().astype(np.float64)
        assert max_err(got, ref) <= TOL[kv]
        assert cache_bytes_equal(dw, oc)
