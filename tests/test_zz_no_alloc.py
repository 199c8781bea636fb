"""pkv_decode_attn_noalloc: decode for callers that cannot allocate device memory.

Programs that embed the library inside an engine whose pool owns all device memory, or
that forbid allocation after start-up, cannot hand the library a workspace; this entry
point keeps its split-K scratch in a fixed array inside the library instead.  The tests
call it through the C ABI on workloads whose automatic plan splits sequences across
blocks (so the scratch is really used), twice in a row (the array keeps the previous
call's contents), and compare with pkv_decode_attn given a caller workspace.  The file
name sorts last so that a stop-at-first-failure run has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {W.F32: 1e-4, W.BF16: 2e-3, W.INT8: 2e-3}
CASES = [
    dict(num_q_heads=8, num_kv_heads=1, head_dim=64, kv_dtype=W.INT8, q_dtype=W.F32,
         decode_lens=[16 * 300 - 3, 16 * 120 + 5]),
    dict(num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16, q_dtype=W.BF16,
         decode_lens=[16 * 400, 1000, 17]),
    dict(num_q_heads=9, num_kv_heads=3, head_dim=64, kv_dtype=W.F32, q_dtype=W.F32,
         decode_lens=[16 * 200 - 1, 333]),
]


def _noalloc(dw, b, out, status):
    """Call the entry point through the C ABI (ctypes, device pointers)."""
    lib = pkv.load()
    c = dw.cache.struct()
    return lib.pkv_decode_attn_noalloc(
        ctypes.byref(c), ctypes.c_void_p(b.q.data_ptr()), pkv._CODE[b.q.dtype], b.q.shape[0],
        b.q.shape[1], ctypes.c_void_p(b.block_tables.data_ptr()), b.block_tables.shape[1],
        ctypes.c_void_p(b.context_lens.data_ptr()), ctypes.c_float(dw.wl.scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_matches_workspace_entry_on_two_calls(case):
    pkv.pkv_set_decode_chunk_pages(0)
    wl = W.small_workload(4000 + case, **CASES[case])
    dw = runner.upload(wl)
    b = dw.batches[0]
    assert b.workspace is not None, "the automatic plan must split so that scratch is used"
    runner.run_batch(dw, 0)  # pkv_decode_attn with a caller workspace
    torch.cuda.synchronize()
    ref = b.out.cpu().numpy().astype(np.float64)
    assert int(dw.dev_status.item()) == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(b.out, float("nan"))
        assert _noalloc(dw, b, out, status) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert int(status.item()) == 0
        assert np.all(np.isfinite(got)), f"call {call}"
        assert float(np.max(np.abs(got - ref))) <= TOL[wl.kv_dtype], f"call {call}"


def test_noalloc_rejects_scratch_beyond_its_maximum():
    wl = W.small_workload(4100, num_q_heads=8, num_kv_heads=1, head_dim=64, kv_dtype=W.INT8,
                          q_dtype=W.F32, decode_lens=[16 * 300] * 8)
    pkv.pkv_set_decode_chunk_pages(1)  # one page per block: 300 splits of 8 sequences x 8 heads
    try:
        dw = runner.upload(wl)
        b = dw.batches[0]
        need = pkv.pkv_decode_workspace_size(dw.cache, 8, 8, b.block_tables.shape[1])
        assert need > pkv.NOALLOC_SCRATCH_BYTES
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.zeros_like(b.out)
        assert _noalloc(dw, b, out, status) == 6  # PKV_ERR_WORKSPACE, nothing launched
        torch.cuda.synchronize()
        assert not out.any()
    finally:
        pkv.pkv_set_decode_chunk_pages(0)
