"""The C ABI without a GPU: the library loads, exports every function include/pkv.h
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from paged_kv_attention_09_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkv.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(pkv.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in pkv.STATUS.items():
        assert pkv.pkv_status_string(code).startswith(name)
    assert pkv.pkv_status_string(1234) == "PKV_UNKNOWN_STATUS"


def _cache(**kw):
    base = dict(k_cache=0x10000, v_cache=0x20000, k_scale=0x30000, v_scale=0x40000,
                num_pages=8, page_size=16, num_kv_heads=2, head_dim=64, kv_dtype=pkv.BF16)
    base.update(kw)
    return pkv.pkv_cache(**base)


def _append(lib, c, k=0x50000, v=0x60000, new_dtype=pkv.F32, slots=0x70000, n=4):
    return lib.pkv_append(ctypes.byref(c) if c is not None else None, k, v, new_dtype, slots, n,
                          None, None)


def test_host_validation_codes(lib):
    assert _append(lib, None) == 1                                  # NULL cache
    assert _append(lib, _cache(k_cache=None)) == 1                  # NULL k_cache
    assert _append(lib, _cache(kv_dtype=7)) == 3                    # dtype
    assert _append(lib, _cache(page_size=8)) == 4                   # page size
    assert _append(lib, _cache(head_dim=96)) == 7                   # unsupported D
    assert _append(lib, _cache(num_pages=0)) == 2                   # shape
    assert _append(lib, _cache(window=-1)) == 2                     # negative window
    assert _append(lib, _cache(k_cache=0x10008)) == 5               # alignment
    assert _append(lib, _cache(kv_dtype=pkv.INT8, k_scale=None)) == 1
    assert _append(lib, _cache(), new_dtype=pkv.INT8) == 3          # INT8 sources
    assert _append(lib, _cache(), k=0x50004) == 5
    assert _append(lib, _cache(), n=-1) == 2
    assert _append(lib, _cache(), k=None, n=0) == 0                 # empty call: no-op


def test_decode_and_prefill_validation(lib):
    c = _cache()
    P = None
    n = ctypes.c_size_t(0)
    # Hq not a multiple of Hkv
    assert lib.pkv_decode_attn(ctypes.byref(c), 0x80000, pkv.F32, 2, 3, 0x90000, 4, 0xA0000,
                               0.1, 0xB0000, P, 0, P, P) == 2
    assert lib.pkv_decode_workspace_size(ctypes.byref(c), 2, 3, 4, ctypes.byref(n)) == 2
    # bad q dtype
    assert lib.pkv_decode_attn(ctypes.byref(c), 0x80000, pkv.INT8, 2, 4, 0x90000, 4, 0xA0000,
                               0.1, 0xB0000, P, 0, P, P) == 3
    # zero sequences: no-op
    assert lib.pkv_decode_attn(ctypes.byref(c), P, pkv.F32, 0, 4, P, 4, P, 0.1, P, P, 0, P,
                               P) == 0
    # misaligned output
    assert lib.pkv_decode_attn(ctypes.byref(c), 0x80000, pkv.F32, 2, 4, 0x90000, 4, 0xA0000,
                               0.1, 0xB0004, P, 0, P, P) == 5
    # max_blocks_per_seq < 1
    assert lib.pkv_decode_attn(ctypes.byref(c), 0x80000, pkv.F32, 2, 4, 0x90000, 0, 0xA0000,
                               0.1, 0xB0000, P, 0, P, P) == 2
    # prefill: negative max_q_len, misaligned q
    assert lib.pkv_prefill_chunk_attn(ctypes.byref(c), 0x80000, pkv.BF16, 2, 4, 0xC0000, -1,
                                      0x90000, 4, 0xA0000, 0.1, 0xB0000, P, 0, P, P) == 2
    assert lib.pkv_prefill_chunk_attn(ctypes.byref(c), 0x80008, pkv.BF16, 2, 4, 0xC0000, 8,
                                      0x90000, 4, 0xA0000, 0.1, 0xB0000, P, 0, P, P) == 5
    assert lib.pkv_decode_workspace_size(ctypes.byref(c), 2, 4, 4, None) == 1


@pytest.mark.parametrize("key_split", [4, -1])
def test_prefill_options_out_of_range(lib, key_split):
    """pkv_prefill_opts.key_split outside 0..3: PKV_ERR_SHAPE from both prefill _ex calls,
    before any device work."""
    c = _cache()
    P = None
    n = ctypes.c_size_t(0)
    o = ctypes.byref(pkv.pkv_prefill_opts(key_split))
    assert lib.pkv_prefill_workspace_size_ex(ctypes.byref(c), 2, 4, 8, 4, o, ctypes.byref(n)) == 2
    assert lib.pkv_prefill_chunk_attn_ex(ctypes.byref(c), 0x80000, pkv.BF16, 2, 4, 0xC0000, 8,
                                         0x90000, 4, 0xA0000, 0.1, 0xB0000, P, 0, o, P, P) == 2


def test_no_device_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = _cache()
    n = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_size(ctypes.byref(c), 2, 4, 4, ctypes.byref(n)) == 9


def test_graph_descriptor_validation(lib):
    """The decode-graph executor rejects bad descriptors on the host."""
    n = ctypes.c_size_t(0)
    h = ctypes.c_void_p(None)
    assert lib.pkv_decode_graph_workspace_size(None, ctypes.byref(n)) == 1
    assert lib.pkv_decode_graph_create(None, ctypes.byref(h)) == 1 and not h.value
    layer = (pkv.pkv_graph_layer * 1)(pkv.pkv_graph_layer(_cache(), 0x80000, 0x90000,
                                                           0x90000, 0xB0000))

    def desc(**kw):
        d = pkv.pkv_decode_graph_desc()
        d.num_layers, d.layers = 1, ctypes.cast(layer, ctypes.POINTER(pkv.pkv_graph_layer))
        d.num_q_heads, d.q_dtype, d.new_dtype = 4, pkv.F32, pkv.F32
        d.block_tables, d.max_blocks_per_seq, d.context_lens = 0xA0000, 4, 0xA1000
        d.slot_mapping = 0xA2000
        b = (ctypes.c_int32 * 3)(1, 2, 4)
        d.num_buckets, d.buckets = 3, ctypes.cast(b, ctypes.POINTER(ctypes.c_int32))
        d._b = b
        for k, v in kw.items():
            setattr(d, k, v)
        return d
    for bad, code in [(dict(num_layers=0), 2), (dict(num_buckets=0), 2),
                      (dict(num_buckets=17), 2), (dict(slot_mapping=None), 1)]:
        d = desc(**bad)
        assert lib.pkv_decode_graph_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code, bad
        assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == code, bad
    d = desc()
    unordered = (ctypes.c_int32 * 3)(1, 4, 2)
    d.buckets = ctypes.cast(unordered, ctypes.POINTER(ctypes.c_int32))
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 2
    layer[0].cache.kv_dtype = 9  # a layer's cache is validated like any call's
    assert lib.pkv_decode_graph_create(ctypes.byref(desc()), ctypes.byref(h)) == 3
    assert lib.pkv_decode_graph_launch(None, 1, None) == 1
    assert lib.pkv_decode_graph_bucket(None, 3) == 0
    lib.pkv_decode_graph_destroy(None)  # a no-op


def test_decode_entry_points_validate_alike(lib):
    """pkv_decode_attn, its _ex form and the no-allocation entry point reject the same
    arguments with the same codes before touching CUDA: among them a block table or a
    page pool too large for 32-bit token positions."""
    P = None
    ok = dict(num_pages=8)

    def calls(c, mb=4, hq=4, q=0x80000, qd=pkv.F32, out=0xB0000, opts=None):
        o = ctypes.byref(opts) if opts is not None else None
        return [
            lib.pkv_decode_attn(ctypes.byref(c), q, qd, 2, hq, 0x90000, mb, 0xA0000, 0.1, out,
                                P, 0, P, P),
            lib.pkv_decode_attn_ex(ctypes.byref(c), q, qd, 2, hq, 0x90000, mb, 0xA0000, 0.1, out,
                                   P, 0, o, P, P),
            lib.pkv_decode_attn_noalloc(ctypes.byref(c), q, qd, 2, hq, 0x90000, mb, 0xA0000, 0.1,
                                        out, P, P),
            lib.pkv_decode_attn_noalloc_ex(ctypes.byref(c), q, qd, 2, hq, 0x90000, mb, 0xA0000,
                                           0.1, out, o, P, P),
        ]
    huge_mb = 0x7fffffff // 16 + 1                            # mb * 16 overflows int32
    assert calls(_cache(**ok), mb=huge_mb) == [2, 2, 2, 2]
    assert calls(_cache(num_pages=0x7fffffff // 16 + 1)) == [2, 2, 2, 2]
    assert calls(_cache(**ok), hq=3) == [2, 2, 2, 2]             # Hq % Hkv
    assert calls(_cache(**ok), qd=pkv.INT8) == [3, 3, 3, 3]      # q dtype
    assert calls(_cache(**ok), out=0xB0004) == [5, 5, 5, 5]      # alignment
    assert calls(_cache(**ok), q=None) == [1, 1, 1, 1]
    assert calls(_cache(kv_dtype=pkv.INT8, k_scale=None)) == [1, 1, 1, 1]
    # a negative split is invalid; the forms without options cannot pass one
    assert calls(_cache(**ok), opts=pkv.pkv_decode_opts(-1))[1::2] == [2, 2]
    n = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_size(ctypes.byref(_cache()), 2, 4, huge_mb,
                                         ctypes.byref(n)) == 2
    assert lib.pkv_decode_workspace_size_ex(ctypes.byref(_cache()), 2, 4, 4,
                                            ctypes.byref(pkv.pkv_decode_opts(-3)),
                                            ctypes.byref(n)) == 2


def test_product_library_has_no_test_hooks(lib):
    """The give-up-at-once wait used by the timeout test exists only in test builds."""
    assert not hasattr(lib, "pkv_test_fail_first_wait")
    assert not hasattr(lib, "pkv_test_prefill_fail_first_wait")
