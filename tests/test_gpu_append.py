"""KV append on the GPU vs the oracle: bit-exact cache contents (slot placement, BF16
rounding, INT8 / FP8 / INT4 codes and scales), skipped padding slots, untouched bytes, bad
slots."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import cache_bytes_equal

pytestmark = pytest.mark.gpu

COMBOS = [(kv, new, D) for kv, new in [(W.F32, W.F32), (W.F32, W.BF16), (W.BF16, W.BF16),
                                      (W.BF16, W.F32), (W.INT8, W.F32), (W.INT8, W.BF16),
                                      (W.FP8, W.F32), (W.FP8, W.BF16), (W.INT4, W.F32),
                                      (W.INT4, W.BF16)]
          for D in (64, 128)]


def _sentinel_caches(wl, value):
    oc = oracle.HostCache(wl.kv_dtype, wl.num_pages, 16, wl.num_kv_heads, wl.head_dim)
    gc = pkv.KVCache.allocate(wl.num_pages, wl.num_kv_heads, wl.head_dim, wl.kv_dtype)
    if wl.kv_dtype in (W.INT8, W.FP8, W.INT4):  # raw bytes: a fixed sentinel pattern
        oc.k[...] = 0xA5
        oc.v[...] = 0xA5
        oc.k_scale[...] = 0.5
        oc.v_scale[...] = 0.5
        gc.k.fill_(0xA5)
        gc.v.fill_(0xA5)
        gc.k_scale.fill_(0.5)
        gc.v_scale.fill_(0.5)
    elif wl.kv_dtype == W.INT8:
        oc.k[...] = value
        oc.v[...] = value
        oc.k_scale[...] = 0.5
        oc.v_scale[...] = 0.5
        gc.k.fill_(value)
        gc.v.fill_(value)
        gc.k_scale.fill_(0.5)
        gc.v_scale.fill_(0.5)
    elif wl.kv_dtype == W.BF16:
        bits = np.uint16(oracle.f32_to_bf16([value])[0])
        oc.k[...] = bits
        oc.v[...] = bits
        gc.k.fill_(value)
        gc.v.fill_(value)
    else:
        oc.k[...] = value
        oc.v[...] = value
        gc.k.fill_(value)
        gc.v.fill_(value)
    return oc, gc


@pytest.mark.parametrize("kv,new,D", COMBOS)
def test_append_bit_exact_with_padding_slots(kv, new, D):
    wl = W.small_workload(40 + D, num_q_heads=4, num_kv_heads=2, head_dim=D, kv_dtype=kv,
                          q_dtype=W.F32, new_dtype=new, decode_lens=[1, 37, 64, 5])
    oc, gc = _sentinel_caches(wl, -3.0)
    slots = wl.slots.copy()
    slots[::7] = -1  # padding tokens
    oracle.append(oc, wl.k_src, wl.v_src, new, slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_append(gc, runner.np_to_torch(wl.k_src).cuda(), runner.np_to_torch(wl.v_src).cuda(),
                   torch.from_numpy(slots).cuda(), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    class DW:
        cache = gc
    assert cache_bytes_equal(DW, oc)


def test_append_int8_extreme_rows():
    """All-zero rows, one-hot rows, huge and subnormal magnitudes, exact ties."""
    D, T = 64, 8
    x = np.zeros((T, 1, D), np.float32)
    x[1, 0, 5] = -3.0                       # one-hot: code -127, others 0
    x[2, 0] = np.linspace(-1e30, 1e30, D)   # huge
    x[3, 0] = np.linspace(-1e-40, 1e-40, D)  # subnormal inputs
    x[4, 0, 0] = 127.0                      # s == 1: exact ties below
    x[4, 0, 1:7] = [2.5, 3.5, -2.5, -3.5, 0.5, -0.5]
    x[5, 0] = np.random.default_rng(0).standard_normal(D) * 1e-3
    x[6, 0] = -np.abs(np.random.default_rng(1).standard_normal(D))
    x[7, 0] = np.float32(1.0) / np.arange(1, D + 1, dtype=np.float32)
    slots = np.arange(T, dtype=np.int32) * 3
    oc = oracle.HostCache(W.INT8, 2, 16, 1, D)
    oracle.append(oc, x, x[::-1].copy(), W.F32, slots)
    gc = pkv.KVCache.allocate(2, 1, D, W.INT8)
    xt = torch.from_numpy(x).cuda()
    pkv.pkv_append(gc, xt, torch.from_numpy(x[::-1].copy()).cuda(), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()

    class DW:
        cache = gc
    assert cache_bytes_equal(DW, oc)


@pytest.mark.parametrize("kv", [W.FP8, W.INT4])
def test_append_fp8_int4_extreme_rows(kv):
    """All-zero rows, one-hot rows, huge and subnormal magnitudes, exact ties (scale 1)."""
    D, T = 64, 8
    x = np.zeros((T, 1, D), np.float32)
    x[1, 0, 5] = -3.0
    x[2, 0] = np.linspace(-1e30, 1e30, D)
    x[3, 0] = np.linspace(-1e-40, 1e-40, D)
    if kv == W.FP8:  # max 448 -> s = 1; E4M3 midpoints (normal and subnormal) round to even
        x[4, 0, :9] = [448.0, 1.0625, 1.1875, 17.0, -17.0, 2.0 ** -10, 3 * 2.0 ** -10,
                       -(2.0 ** -10), 0.0]
    else:            # max 7 -> s = 1; halves round to even
        x[4, 0, :8] = [7.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, 6.5]
    x[5, 0] = np.random.default_rng(0).standard_normal(D) * 1e-3
    x[6, 0] = -np.abs(np.random.default_rng(1).standard_normal(D))
    x[7, 0] = np.float32(1.0) / np.arange(1, D + 1, dtype=np.float32)
    slots = np.arange(T, dtype=np.int32) * 3
    oc = oracle.HostCache(kv, 2, 16, 1, D)
    oracle.append(oc, x, x[::-1].copy(), W.F32, slots)
    gc = pkv.KVCache.allocate(2, 1, D, kv)
    pkv.pkv_append(gc, torch.from_numpy(x).cuda(), torch.from_numpy(x[::-1].copy()).cuda(),
                   torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()

    class DW:
        cache = gc
    assert cache_bytes_equal(DW, oc)


def test_append_int4_many_tokens_of_one_page():
    """Every token of several pages in one call: INT4 V bytes are per token, so concurrent
    appends into one page must not disturb each other."""
    wl = W.small_workload(55, num_q_heads=4, num_kv_heads=2, head_dim=128, kv_dtype=W.INT4,
                          q_dtype=W.F32, decode_lens=[64, 48, 16])
    oc, gc = _sentinel_caches(wl, 0.0)
    oracle.append(oc, wl.k_src, wl.v_src, W.F32, wl.slots)
    pkv.pkv_append(gc, runner.np_to_torch(wl.k_src).cuda(), runner.np_to_torch(wl.v_src).cuda(),
                   torch.from_numpy(wl.slots).cuda())
    torch.cuda.synchronize()

    class DW:
        cache = gc
    assert cache_bytes_equal(DW, oc)


def test_append_bad_slot_sets_status_and_is_skipped():
    wl = W.small_workload(50, num_q_heads=2, num_kv_heads=2, head_dim=64, kv_dtype=W.BF16,
                          q_dtype=W.BF16, decode_lens=[20])
    oc, gc = _sentinel_caches(wl, 1.0)
    slots = wl.slots.copy()
    slots[3] = wl.num_pages * 16 + 1
    oracle.append(oc, wl.k_src, wl.v_src, W.BF16, slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_append(gc, runner.np_to_torch(wl.k_src).cuda(), runner.np_to_torch(wl.v_src).cuda(),
                   torch.from_numpy(slots).cuda(), status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkv.DEV_BAD_SLOT

    class DW:
        cache = gc
    assert cache_bytes_equal(DW, oc)


@pytest.mark.parametrize("name", ["tiny", "smollm2-f32", "qwen-bf16", "tinyllama-int8",
                                  "tinyllama-fp8", "tinyllama-int4"])
def test_full_size_cache_bit_exact(name):
    """The whole cache after the history and the step's appends, at full size."""
    wl = W.workload(name)
    dw = runner.upload(wl, "cuda")
    runner.append_rows(dw, dw.step_rows)
    torch.cuda.synchronize()
    assert int(dw.dev_status.item()) == 0
    oc = oracle.cache_from_workload(wl)
    assert cache_bytes_equal(dw, oc)
