"""Prefix-shared pages ("tinyloop Current Status", KV cache modes table: prefix caching):
several block tables alias the same physical pages.  Decode, prefill and the fused decode
step on the GPU vs the oracle, with sequences that share their first pages."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import TOL, max_err

pytestmark = pytest.mark.gpu


def share_prefix(bt, lens, pairs):
    """Sequence b2 reads the first n pages of sequence b1 (whose content was written
    through b1's table); returns the edited table."""
    bt = bt.copy()
    for b1, b2, n in pairs:
        assert n * 16 <= min(lens[b1], lens[b2])
        bt[b2, :n] = bt[b1, :n]
    return bt


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8])
def test_decode_with_shared_prefix_pages(kv):
    wl = W.small_workload(7300 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[200, 180, 97, 300])
    b = wl.batches[0]
    # 1 and 3 share 5 and 11 pages of sequence 0's prefix; 2 shares 6 pages of 1's
    # (which are themselves 0's first 5 pages plus one of its own)
    bt = share_prefix(b.block_tables, b.context_lens, [(0, 1, 5), (0, 3, 11), (1, 2, 6)])
    oc = oracle.cache_from_workload(wl)
    ref = oracle.decode(oc, b.q, b.q_dtype, bt, b.context_lens, wl.scale)
    dw = runner.upload(wl, "cuda")
    runner.append_rows(dw, dw.step_rows)
    db = dw.batches[0]
    db.block_tables.copy_(torch.from_numpy(bt))
    for chunk in (0, 2):  # automatic split, and a forced split so shared pages cross blocks
        dw.split_pages = chunk
        db.workspace = pkv.workspace_for(pkv.pkv_decode_workspace_size(
            dw.cache, b.num_seqs, wl.num_q_heads, b.max_blocks, chunk), "cuda")
        runner.run_batch(dw, 0)
        torch.cuda.synchronize()
        assert int(dw.dev_status.item()) == 0
        got = db.out.cpu().numpy().astype(np.float64)
        assert max_err(got, ref) <= TOL[kv]


def test_prefill_chunks_over_shared_prefix():
    """Two prompts continue from one cached prefix (same physical pages)."""
    wl = W.small_workload(7310, num_q_heads=12, num_kv_heads=2, head_dim=128, kv_dtype=W.BF16,
                          q_dtype=W.BF16, prefill=[(96, 40), (96, 70)])
    b = wl.batches[0]
    bt = share_prefix(b.block_tables, b.context_lens, [(0, 1, 6)])  # the 96-token prefix
    oc = oracle.cache_from_workload(wl)
    ref = oracle.prefill(oc, b.q, b.q_dtype, b.q_start_loc, bt, b.context_lens, wl.scale)
    dw = runner.upload(wl, "cuda")
    runner.append_rows(dw, dw.step_rows)
    dw.batches[0].block_tables.copy_(torch.from_numpy(bt))
    runner.run_batch(dw, 0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    assert max_err(got, ref) <= TOL[W.BF16]


@pytest.mark.parametrize("kv", [W.BF16, W.INT8])
def test_fused_step_with_shared_prefix(kv):
    """New tokens go into each sequence's own last page while the prefix pages are shared."""
    wl = W.small_workload(7320 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[100, 90, 130])
    b = wl.batches[0]
    bt = share_prefix(b.block_tables, b.context_lens, [(0, 1, 4), (0, 2, 5)])
    rows = wl.step_rows[:b.num_seqs]
    pos = (b.context_lens - 1).astype(np.int32)
    oc = oracle.cache_from_workload(wl, rows=wl.history_rows)
    slots = np.array([bt[s, (int(b.context_lens[s]) - 1) // 16] * 16 + (int(b.context_lens[s]) - 1) % 16
                      for s in range(b.num_seqs)], np.int32)
    ref = oracle.decode_step(oc, b.q, b.q_dtype, wl.k_src[rows], wl.v_src[rows], wl.new_dtype,
                             slots, pos, 10000.0, bt, b.context_lens, wl.scale)
    dw = runner.upload(wl, "cuda")
    dw.batches[0].block_tables.copy_(torch.from_numpy(bt))
    k, v, _, p = runner.decode_step_inputs(dw, 0, True)
    runner.run_decode_step(dw, (k, v, torch.from_numpy(slots).cuda(), p), 0, 10000.0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    assert max_err(got, ref) <= TOL[kv]
