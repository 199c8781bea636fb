"""pkv_decode_attn_noalloc: decode for callers that cannot allocate device memory.

Programs that embed the library inside an engine whose pool owns all device memory, or
that forbid allocation after start-up, cannot hand the library a workspace; this entry
point keeps its split-K scratch in a fixed array inside the library instead.  The tests
call it through the C ABI on workloads whose plan splits sequences across more blocks
than merge on chip (so the scratch is really used), twice in a row (the array keeps the
previous call's contents), and require the result of pkv_decode_attn with a caller
workspace bit for bit: both run the same plan and kernel.  The file name sorts last so
that a stop-at-first-failure run has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {W.F32: 1e-4, W.BF16: 2e-3, W.INT8: 2e-3, W.FP8: 2e-3, W.INT4: 2e-3}
CASES = [
    dict(num_q_heads=8, num_kv_heads=1, head_dim=64, kv_dtype=W.INT8, q_dtype=W.F32,
         decode_lens=[16 * 300 - 3, 16 * 120 + 5]),
    dict(num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16, q_dtype=W.BF16,
         decode_lens=[16 * 400, 1000, 17]),
    dict(num_q_heads=9, num_kv_heads=3, head_dim=64, kv_dtype=W.F32, q_dtype=W.F32,
         decode_lens=[16 * 200 - 1, 333]),
    dict(num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=W.FP8, q_dtype=W.F32,
         decode_lens=[16 * 260 + 7, 900]),
    dict(num_q_heads=16, num_kv_heads=2, head_dim=128, kv_dtype=W.INT4, q_dtype=W.BF16,
         decode_lens=[16 * 280 - 9, 40]),
]


def _noalloc(dw, b, out, status, split_pages=0):
    """Call the entry point through the C ABI (ctypes, device pointers); split_pages > 0
    goes through the _ex form with that option."""
    lib = pkv.load()
    c = dw.cache.struct()
    args = [ctypes.byref(c), ctypes.c_void_p(b.q.data_ptr()), pkv._CODE[b.q.dtype],
            b.q.shape[0], b.q.shape[1], ctypes.c_void_p(b.block_tables.data_ptr()),
            b.block_tables.shape[1], ctypes.c_void_p(b.context_lens.data_ptr()),
            ctypes.c_float(dw.wl.scale), ctypes.c_void_p(out.data_ptr())]
    tail = [ctypes.c_void_p(status.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]
    if split_pages:
        opts = pkv.pkv_decode_opts(split_pages)
        return lib.pkv_decode_attn_noalloc_ex(*args, ctypes.byref(opts), *tail)
    return lib.pkv_decode_attn_noalloc(*args, *tail)


def _both(dw, b, split_pages=0):
    """pkv_decode_attn's output with a caller workspace, then two no-allocation calls;
    returns (reference, [outputs of the two calls])."""
    runner.run_batch(dw, 0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    ref = b.out.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = []
    for call in range(2):
        out = torch.full_like(b.out, float("nan"))
        assert _noalloc(dw, b, out, status, split_pages) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}"
        got.append(out.cpu().numpy())
    return ref, got


@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_matches_workspace_entry_on_two_calls(case):
    wl = W.small_workload(4000 + case, **CASES[case])
    dw = runner.upload(wl, split_pages=16)  # >= 13 splits: merged through the scratch
    b = dw.batches[0]
    assert b.workspace is not None, "the plan must use scratch"
    ref, got = _both(dw, b, split_pages=16)
    for call, g in enumerate(got):
        assert np.all(np.isfinite(g)), f"call {call}"
        assert np.array_equal(g, ref), f"call {call}: not bit-identical to pkv_decode_attn"
        err = float(np.max(np.abs(g.astype(np.float64) - ref.astype(np.float64))))
        assert err <= TOL[wl.kv_dtype]


def _bracket_workload(pages):
    """16 INT8 sequences of 32 q / 4 kv heads over `pages`-wide block tables: with one page
    per block the split scratch is 256 + pages * 16 * 32 * 66 * 4 bytes, just under the
    4 MiB maximum at 31 pages and just over it at 32."""
    return W.small_workload(4100 + pages, num_q_heads=32, num_kv_heads=4, head_dim=64,
                            kv_dtype=W.INT8, q_dtype=W.F32,
                            decode_lens=[16 * pages - (s % 5) for s in range(16)],
                            max_decode_len=16 * pages)


def test_noalloc_at_its_maximum_matches_workspace_entry():
    wl = _bracket_workload(31)
    dw = runner.upload(wl, split_pages=1)
    b = dw.batches[0]
    need = pkv.pkv_decode_workspace_size(dw.cache, 16, 32, b.block_tables.shape[1], 1)
    assert need == 256 + 31 * 16 * 32 * 66 * 4
    assert pkv.NOALLOC_SCRATCH_BYTES - 4096 < need <= pkv.NOALLOC_SCRATCH_BYTES
    ref, got = _both(dw, b, split_pages=1)
    for call, g in enumerate(got):
        assert np.array_equal(g, ref), f"call {call}: not bit-identical to pkv_decode_attn"


def test_noalloc_rejects_scratch_beyond_its_maximum():
    wl = _bracket_workload(32)
    dw = runner.upload(wl, split_pages=1)
    b = dw.batches[0]
    need = pkv.pkv_decode_workspace_size(dw.cache, 16, 32, b.block_tables.shape[1], 1)
    assert pkv.NOALLOC_SCRATCH_BYTES < need < pkv.NOALLOC_SCRATCH_BYTES + 256 * 1024
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(b.out)
    assert _noalloc(dw, b, out, status, split_pages=1) == 6  # PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any(), "nothing may be launched"
    assert int(status.item()) == 0


def test_noalloc_with_an_on_chip_merge_needs_no_scratch():
    """A sequence split over at most 8 blocks merges on chip: no workspace is needed, and
    the no-allocation entry point gives pkv_decode_attn's result bit for bit."""
    wl = W.small_workload(4200, num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, decode_lens=[16 * 64, 16 * 30 + 3, 5])
    dw = runner.upload(wl, split_pages=8)  # 8 splits of the 64-page table
    b = dw.batches[0]
    assert pkv.pkv_decode_workspace_size(dw.cache, 3, 12, b.block_tables.shape[1], 8) == 0
    ref, got = _both(dw, b, split_pages=8)
    for call, g in enumerate(got):
        assert np.array_equal(g, ref), f"call {call}"
