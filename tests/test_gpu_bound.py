"""pkv.BoundCall: a library call marshalled once and issued again without the wrapper.

A loop that repeats the same launches on fixed buffers (a serving step, the benchmark's
end-to-end leg) binds each call once and re-issues it with nothing but the ctypes call.
The bound form must be the same C call: every launch kind (append, decode, chunked
prefill, fused decode step) bound and issued twice gives the wrapper's output and cache
bit for bit, and a bound call whose status is an error raises like the wrapper.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _snapshot(dw):
    return [b.out.cpu().clone() for b in dw.batches], dw.cache.k.cpu().clone(), \
        dw.cache.v.cpu().clone()


@pytest.mark.parametrize("kv", [W.BF16, W.INT8])
def test_bound_append_decode_prefill_match_wrappers(kv):
    wl = W.small_workload(40 + kv, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                          q_dtype=W.F32, decode_lens=[16 * 30 + 5, 77],
                          prefill=[(50, 20)] if kv == W.BF16 else ())
    # the wrappers
    dw = runner.upload(wl, "cuda", split_pages=4)
    rows = dw.step_rows
    k, v, s = dw.k_src[rows], dw.v_src[rows], dw.slots[rows]
    pkv.pkv_append(dw.cache, k, v, s, dw.dev_status)
    for j in range(len(dw.batches)):
        runner.run_batch(dw, j)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    outs, kc, vc = _snapshot(dw)
    # the same calls bound, on a fresh upload, issued twice
    dw2 = runner.upload(wl, "cuda", split_pages=4)
    k2, v2, s2 = dw2.k_src[rows], dw2.v_src[rows], dw2.slots[rows]
    calls = [pkv.pkv_append(dw2.cache, k2, v2, s2, dw2.dev_status, bound=True)]
    calls += [runner.run_batch(dw2, j, bound=True) for j in range(len(dw2.batches))]
    assert all(isinstance(c, pkv.BoundCall) for c in calls)
    for b in dw2.batches:
        b.out.fill_(float("nan"))  # nothing ran at bind time
    for _ in range(2):
        for c in calls:
            c()
    torch.cuda.synchronize()
    assert int(dw2.dev_status.item()) == 0
    outs2, kc2, vc2 = _snapshot(dw2)
    for a, b in zip(outs, outs2):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(kc.view(torch.uint8), kc2.view(torch.uint8))
    assert torch.equal(vc.view(torch.uint8), vc2.view(torch.uint8))


def test_bound_fused_step_matches_wrapper():
    wl = W.small_workload(45, num_q_heads=8, num_kv_heads=1, head_dim=64, kv_dtype=W.INT8,
                          q_dtype=W.F32, decode_lens=[16 * 20 + 1, 300, 16])
    dw = runner.upload(wl, "cuda")
    inp = runner.decode_step_inputs(dw, 0, True)
    runner.run_decode_step(dw, inp, 0, 10000.0)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    outs, kc, vc = _snapshot(dw)
    dw2 = runner.upload(wl, "cuda")
    inp2 = runner.decode_step_inputs(dw2, 0, True)
    call = runner.run_decode_step(dw2, inp2, 0, 10000.0, bound=True)
    dw2.batches[0].out.fill_(float("nan"))
    call()
    call()  # the new row lands at the same slot again: same cache, same output
    torch.cuda.synchronize()
    assert int(dw2.dev_status.item()) == 0
    outs2, kc2, vc2 = _snapshot(dw2)
    assert torch.equal(outs[0].view(torch.uint8), outs2[0].view(torch.uint8))
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)


def test_bound_call_raises_on_error_status():
    wl = W.small_workload(46, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=W.F32,
                          q_dtype=W.F32, decode_lens=[40])
    dw = runner.upload(wl, "cuda")
    b = dw.batches[0]
    null_out = torch.empty(0, device="cuda")  # an empty tensor has no storage: a null pointer
    assert null_out.data_ptr() == 0
    call = pkv.pkv_decode_attn(dw.cache, b.q, b.block_tables, b.context_lens, wl.scale,
                               null_out, None, dw.dev_status, bound=True)
    with pytest.raises(pkv.PkvError) as e:
        call()
    assert e.value.code == 1  # PKV_ERR_NULL
    np.testing.assert_equal(int(dw.dev_status.item()), 0)
