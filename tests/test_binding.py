"""The Python binding's host logic without a GPU: bound calls (pkv.BoundCall).

A wrapper called with bound=True marshals its arguments and returns the call without
issuing it; calling the result issues exactly the C call the wrapper would have issued,
as often as it is called, and a non-zero status raises PkvError like the wrapper.  A
recording stand-in for the library checks the calls; the real library checks the status
path (no device here: PKV_ERR_DEVICE).
"""
import ctypes
import os

import pytest
import torch

from paged_kv_attention_09_gb300 import pkv


class _Recorder:
    """Stands in for the library: every pkv_* entry point records its arguments."""

    def __init__(self, code=0):
        self.calls, self.code = [], code

    def __getattr__(self, name):
        if not name.startswith("pkv_"):
            raise AttributeError(name)

        def entry(*args):
            self.calls.append((name, args))
            return self.code
        return entry


def _plain(args):
    """Comparable values of a recorded argument list (pointers, structs, scalars)."""
    out = []
    for a in args:
        if isinstance(a, ctypes.c_void_p):
            out.append(("ptr", a.value))
        elif type(a).__name__ == "CArgObject":  # byref(struct): its fields
            obj = a._obj
            out.append(("struct", tuple(getattr(obj, f) for f, _ in obj._fields_)))
        elif a is None:
            out.append(None)
        else:
            out.append(a)
    return out


def _inputs():
    cache = pkv.KVCache(torch.zeros(8, 2, 16, 64), torch.zeros(8, 2, 64, 16))
    q = torch.zeros(3, 4, 64)
    bt = torch.zeros(3, 2, dtype=torch.int32)
    lens = torch.full((3,), 20, dtype=torch.int32)
    out = torch.zeros(3, 4, 64)
    return cache, q, bt, lens, out


def test_bound_call_issues_the_wrappers_call(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(pkv, "load", lambda path=pkv.LIB_PATH: rec)
    cache, q, bt, lens, out = _inputs()
    pkv.pkv_decode_attn(cache, q, bt, lens, 0.125, out, stream=0, split_pages=2)
    assert len(rec.calls) == 1
    call = pkv.pkv_decode_attn(cache, q, bt, lens, 0.125, out, stream=0, split_pages=2,
                               bound=True)
    assert isinstance(call, pkv.BoundCall)
    assert len(rec.calls) == 1  # nothing issued at bind time
    call()
    call()
    assert len(rec.calls) == 3
    (n0, a0), (n1, a1), (n2, a2) = rec.calls
    assert n0 == n1 == n2 == "pkv_decode_attn_ex"
    p0, p1, p2 = _plain(a0), _plain(a1), _plain(a2)
    opts = [i for i, a in enumerate(a0) if type(a).__name__ == "CArgObject"][1]
    assert a1[opts]._obj.split_pages == 2
    assert p1 == p2 == p0
    assert ("ptr", q.data_ptr()) in p1 and ("ptr", out.data_ptr()) in p1


def test_bound_append_prefill_and_step_are_not_issued_at_bind_time(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(pkv, "load", lambda path=pkv.LIB_PATH: rec)
    cache, q, bt, lens, out = _inputs()
    k = torch.zeros(3, 2, 64)
    slots = torch.zeros(3, dtype=torch.int32)
    loc = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    calls = [pkv.pkv_append(cache, k, k, slots, stream=0, bound=True),
             pkv.pkv_prefill_chunk_attn(cache, q, loc, 1, bt, lens, 0.125, out, stream=0,
                                        bound=True),
             pkv.pkv_decode_step(cache, q, k, k, slots, None, 1e4, bt, lens, 0.125, out,
                                 stream=0, bound=True)]
    assert rec.calls == []
    for c in calls:
        c()
    assert [n for n, _ in rec.calls] == ["pkv_append", "pkv_prefill_chunk_attn_ex",
                                         "pkv_decode_step_ex"]


def test_bound_call_raises_the_status(monkeypatch):
    rec = _Recorder(code=2)
    monkeypatch.setattr(pkv, "load", lambda path=pkv.LIB_PATH: rec)
    cache, q, bt, lens, out = _inputs()
    call = pkv.pkv_decode_attn(cache, q, bt, lens, 0.125, out, stream=0, bound=True)
    with pytest.raises(pkv.PkvError) as e:
        call()
    assert e.value.code == 2 and "PKV_ERR_SHAPE" in str(e.value)


def test_bound_call_reaches_the_library():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    if not os.path.exists(pkv.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    pkv.load()
    cache, q, bt, lens, out = _inputs()
    call = pkv.pkv_decode_attn(cache, q, bt, lens, 0.125, out, stream=0, bound=True)
    with pytest.raises(pkv.PkvError) as e:
        call()
    assert e.value.code == 9  # PKV_ERR_DEVICE: the host checks passed, no device here
