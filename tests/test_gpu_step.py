"""The fused decode step on the GPU (rotary embedding, append of the new row, attention
in one launch) vs the FP64 oracle's decode step: outputs within the dtype tolerance, the
whole cache bit for bit, and the step's own error cases."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import TOL, cache_bytes_equal, max_err

pytestmark = pytest.mark.gpu

THETA = 10000.0


def step_case(seed, kv, qd, nd, Hq, Hkv, D, lens, rope=True, chunk=0, slot_edit=None):
    wl = W.small_workload(seed, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, kv_dtype=kv,
                          q_dtype=qd, new_dtype=nd, decode_lens=lens)
    b = wl.batches[0]
    B = b.num_seqs
    rows = wl.step_rows[:B]
    k_new, v_new = wl.k_src[rows], wl.v_src[rows]
    slots = wl.slots[rows].astype(np.int32).copy()
    if slot_edit is not None:
        slot_edit(slots, wl)
    pos = (b.context_lens - 1).astype(np.int32) if rope else None
    oc = oracle.cache_from_workload(wl, rows=wl.history_rows)
    ref = oracle.decode_step(oc, b.q, qd, k_new, v_new, nd, slots, pos, THETA, b.block_tables,
                             b.context_lens, wl.scale)
    dw = runner.upload(wl, "cuda", split_pages=chunk)
    k, v, _, p = runner.decode_step_inputs(dw, 0, rope)
    runner.run_decode_step(dw, (k, v, torch.from_numpy(slots).cuda(), p), 0, THETA)
    torch.cuda.synchronize()
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    return wl, ref, got, int(dw.dev_status.item()), dw, oc


CASES = [
    # kv, q, new, Hq, Hkv, D, lens
    (W.F32, W.F32, W.F32, 9, 3, 64, [37, 16, 1, 70]),
    (W.F32, W.BF16, W.F32, 8, 2, 128, [33, 100]),
    (W.BF16, W.BF16, W.BF16, 12, 2, 128, [130, 1, 47, 16]),
    (W.BF16, W.F32, W.F32, 8, 8, 64, [5, 64, 65]),
    (W.INT8, W.F32, W.F32, 32, 4, 64, [20, 1, 33, 300]),
    (W.INT8, W.BF16, W.F32, 6, 1, 128, [48, 17]),
    (W.INT8, W.F32, W.BF16, 32, 2, 64, [9, 81]),  # two head groups of 8
    (W.BF16, W.BF16, W.BF16, 32, 2, 128, [77, 3]),  # two head groups of 8
    (W.FP8, W.F32, W.F32, 32, 4, 64, [20, 1, 33, 300]),
    (W.FP8, W.BF16, W.BF16, 6, 1, 128, [48, 17]),
    (W.INT4, W.F32, W.F32, 32, 4, 64, [20, 1, 33, 300]),
    (W.INT4, W.BF16, W.F32, 12, 2, 128, [48, 17, 5]),
]


@pytest.mark.parametrize("rope", [True, False])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_step_matches_oracle(case, rope):
    kv, qd, nd, Hq, Hkv, D, lens = CASES[case]
    wl, ref, got, status, dw, oc = step_case(7000 + case, kv, qd, nd, Hq, Hkv, D, lens, rope)
    assert status == 0
    assert max_err(got, ref) <= TOL[kv]
    assert cache_bytes_equal(dw, oc)  # the new rows stored exactly as the oracle stores them


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_step_with_splits(kv):
    """Long contexts split over several blocks: the block of the last split patches the
    new token; the automatic split and a forced small chunk."""
    for chunk in (0, 3):
        wl, ref, got, status, dw, oc = step_case(7100 + kv, kv, W.F32 if kv != W.BF16 else W.BF16,
                                                 W.F32, 8, 1, 64, [16 * 40 - 3, 16 * 7 + 1, 2],
                                                 True, chunk)
        assert status == 0
        assert max_err(got, ref) <= TOL[kv]
        assert cache_bytes_equal(dw, oc)


@pytest.mark.parametrize("kv", [W.F32, W.BF16, W.INT8, W.FP8, W.INT4])
def test_step_bad_slot_and_no_new_token(kv):
    """Sequence 0's slot is not its last position's slot: NaN rows, status bit, nothing
    stored for it; sequence 1 has no new token (slot -1) and attends over the cache as is;
    sequence 2 is a normal step."""
    def edit(slots, wl):
        slots[0] = (slots[0] + 1) % (wl.num_pages * 16)
        slots[1] = -1
    wl, ref, got, status, dw, oc = step_case(7200 + kv, kv, W.F32, W.F32, 4, 2, 64,
                                             [20, 35, 50], True, 0, edit)
    assert status & pkv.DEV_BAD_SLOT
    assert np.all(np.isnan(got[0]))
    assert np.all(np.isfinite(got[1:]))
    assert max_err(got, ref, [1, 2]) <= TOL[kv]
    assert cache_bytes_equal(dw, oc)


def test_step_bench_config_sampled():
    """The benchmark's INT8 workload as one fused step, sampled sequences vs the oracle."""
    wl = W.workload("tinyllama-int8")
    b = wl.batches[0]
    rows = wl.step_rows[:b.num_seqs]
    dw = runner.upload(wl, "cuda")
    inp = runner.decode_step_inputs(dw, 0, True)
    runner.run_decode_step(dw, inp, 0, THETA)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    got = dw.batches[0].out.cpu().numpy().astype(np.float64)
    seqs = [0, 1, 100, 255]
    oc = oracle.cache_from_workload(wl, rows=wl.history_rows)
    ref = oracle.decode_step(oc, b.q, b.q_dtype, wl.k_src[rows], wl.v_src[rows], wl.new_dtype,
                             wl.slots[rows], (b.context_lens - 1).astype(np.int32), THETA,
                             b.block_tables, b.context_lens, wl.scale, seqs=seqs)
    assert max_err(got, ref, seqs) <= TOL[wl.kv_dtype]
