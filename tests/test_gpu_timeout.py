"""The decode and prefill kernels' bounded waits, when they give up: the call reports
PKV_DEV_TIMEOUT, the affected rows are NaN, every copy in flight is drained before the
block reuses its shared memory or exits, and the next call on the same buffers is clean.

A wait that really runs out needs a copy that never lands, which no correct program
makes; a test build of the library (compiled here with PKV_TEST_HOOKS, never the product
library) therefore lets the first page wait of every decode warp, or the first score
wait of every prefill softmax group, give up at once.  The decode drain keeps its full
limit so that every copy lands before the block moves on; in the prefill the other
roles' waits then run out on their own (bounded) limits, about a second."""
import ctypes
import os

import numpy as np
import pytest
import torch

from paged_kv_attention_09_gb300 import _build, pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks(tmp_path_factory):
    d = tmp_path_factory.mktemp("hooks")
    path = _build.build(defines=["-DPKV_TEST_HOOKS"], lib=os.path.join(str(d), "libpkv_hooks.so"),
                        obj=os.path.join(str(d), "obj"))
    lib = pkv.bind(path)
    for fn in ("pkv_test_fail_first_wait", "pkv_test_prefill_fail_first_wait"):
        getattr(lib, fn).argtypes = [ctypes.c_int]
        getattr(lib, fn).restype = ctypes.c_int
    yield lib
    lib.pkv_test_fail_first_wait(0)
    lib.pkv_test_prefill_fail_first_wait(0)


def _decode(lib, dw, split_pages):
    b = dw.batches[0]
    out = torch.full_like(b.out, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = dw.cache.struct()
    ws = b.workspace
    opts = pkv.pkv_decode_opts(split_pages)
    rc = lib.pkv_decode_attn_ex(
        ctypes.byref(c), ctypes.c_void_p(b.q.data_ptr()), pkv._CODE[b.q.dtype], b.q.shape[0],
        b.q.shape[1], ctypes.c_void_p(b.block_tables.data_ptr()), b.block_tables.shape[1],
        ctypes.c_void_p(b.context_lens.data_ptr()), ctypes.c_float(dw.wl.scale),
        ctypes.c_void_p(out.data_ptr()), None if ws is None else ctypes.c_void_p(ws.data_ptr()),
        0 if ws is None else ws.numel() * ws.element_size(), ctypes.byref(opts),
        ctypes.c_void_p(status.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("kv,D,split", [(W.INT8, 64, 0), (W.INT8, 64, 3), (W.BF16, 128, 4),
                                        (W.F32, 64, 2), (W.FP8, 128, 0), (W.INT4, 64, 5)])
def test_wait_that_gives_up_reports_timeout_then_next_call_is_clean(hooks, kv, D, split):
    wl = W.small_workload(8800 + kv * 10 + split, num_q_heads=8, num_kv_heads=2, head_dim=D,
                          kv_dtype=kv, q_dtype=W.F32, decode_lens=[16 * 20 + 3, 40, 1])
    dw = runner.upload(wl, split_pages=split)
    runner.append_rows(dw, dw.step_rows)
    runner.run_batch(dw, 0)  # the product library's result
    torch.cuda.synchronize()
    ref = dw.batches[0].out.cpu().numpy()
    assert int(dw.dev_status.item()) == 0

    assert hooks.pkv_test_fail_first_wait(1) == 0
    got, status = _decode(hooks, dw, split)
    assert status & pkv.DEV_TIMEOUT
    assert np.all(np.isnan(got)), "every block gave up on its first page: NaN rows"

    assert hooks.pkv_test_fail_first_wait(0) == 0
    for _ in range(2):  # the workspace counters were left ready: the next calls are exact
        got, status = _decode(hooks, dw, split)
        assert status == 0
        assert np.array_equal(got, ref)


def _prefill(lib, dw, key_split):
    b = dw.batches[0]
    out = torch.full_like(b.out, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = dw.cache.struct()
    ws = b.workspace
    opts = pkv.pkv_prefill_opts(key_split)
    rc = lib.pkv_prefill_chunk_attn_ex(
        ctypes.byref(c), ctypes.c_void_p(b.q.data_ptr()), pkv._CODE[b.q.dtype], len(b.context_lens),
        b.q.shape[1], ctypes.c_void_p(b.q_start_loc.data_ptr()), b.max_q_len,
        ctypes.c_void_p(b.block_tables.data_ptr()), b.block_tables.shape[1],
        ctypes.c_void_p(b.context_lens.data_ptr()), ctypes.c_float(dw.wl.scale),
        ctypes.c_void_p(out.data_ptr()), None if ws is None else ctypes.c_void_p(ws.data_ptr()),
        0 if ws is None else ws.numel() * ws.element_size(), ctypes.byref(opts),
        ctypes.c_void_p(status.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("D,qd,key_split", [(128, W.BF16, 1), (64, W.F32, 3)])
def test_prefill_wait_that_gives_up_reports_timeout_then_next_call_is_clean(hooks, D, qd,
                                                                             key_split):
    wl = W.small_workload(8900 + D + key_split, num_q_heads=8, num_kv_heads=2, head_dim=D,
                          kv_dtype=W.BF16, q_dtype=qd, prefill=[(300, 70), (0, 20), (1000, 5)])
    dw = runner.upload(wl, key_split=key_split)
    runner.append_rows(dw, dw.step_rows)
    runner.run_batch(dw, 0)  # the product library's result
    torch.cuda.synchronize()
    ref = dw.batches[0].out.cpu().numpy()
    assert int(dw.dev_status.item()) == 0

    assert hooks.pkv_test_prefill_fail_first_wait(1) == 0
    got, status = _prefill(hooks, dw, key_split)
    assert status & pkv.DEV_TIMEOUT
    assert np.all(np.isnan(got)), "every softmax group gave up on its first scores: NaN rows"

    assert hooks.pkv_test_prefill_fail_first_wait(0) == 0
    for _ in range(2):  # the workspace counters were left ready: the next calls are exact
        got, status = _prefill(hooks, dw, key_split)
        assert status == 0
        assert np.array_equal(got, ref)
