"""Pins for the CPU oracle: each ties it to something other than itself.

- BF16 rounding against torch's float->bfloat16 cast (a library routine) on random
  values and on constructed ties.
- The INT8 quantiser against an exhaustive nearest-code search, hand-made ties, and the
  round-trip bound |x - code*s| <= s/2.
- Attention against torch's scaled_dot_product_attention in float64 on the logically
  reassembled cache (dense brute force), for decode and for causal chunks.
- Closed forms: uniform V, a single token, q = 0, one dominating key.
- Structure: physical page order does not matter; GQA equals MHA with replicated heads;
  causality (future keys do not matter, the last chunk row equals decode, Lq = 1 equals
  decode).
- Planted mistakes: each deliberately broken oracle build fails at least one pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, F32, FP8, INT4, INT8, QUANTISED, HostCache
from paged_kv_attention_09_gb300 import workloads as W

P = 16


# --------------------------------------------------------------------------- helpers

def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def k_elem(dtype, t, d, D):
    """Element index of K (token t, column d) inside one (page, kv head) block."""
    if dtype == BF16:  # tensor-core tiles: 8x8 core matrices of 64 contiguous elements
        return ((t // 8) * (D // 8) + d // 8) * 64 + (t % 8) * 8 + d % 8
    return t * D + d


def v_elem(dtype, t, d, D):
    """Element index of V (token t, column d) inside one (page, kv head) block."""
    if dtype == BF16:
        return ((d // 8) * (P // 8) + t // 8) * 64 + (d % 8) * 8 + t % 8
    return d * P + t


def e4m3_torch(x):
    """float32 -> FP8 E4M3 codes by the library cast (round to nearest even)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def e4m3_decode_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def int4_codes(rows):
    """Unpack INT4 K rows (uint8 [..., n/2]) into codes [..., n] by the documented layout:
    every 8 consecutive elements form a little-endian 32-bit word in which element e sits
    at bit 4 * ((e >> 1) + 4 * (e & 1)); 4-bit two's complement."""
    b = rows.reshape(*rows.shape[:-1], -1, 4).astype(np.uint32)
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    e = np.arange(8, dtype=np.uint32)
    nib = ((word[..., None] >> (4 * ((e >> 1) + 4 * (e & 1)))) & 15).astype(np.int64)
    return np.where(nib >= 8, nib - 16, nib).reshape(*rows.shape[:-1], -1)


def int4_v_codes(v):
    """Unpack an INT4 V cache (uint8 [NP, Hkv, D/2, 16]) into codes [NP, Hkv, D, 16]: row
    pair p holds head-dim rows 16 (p // 8) + p % 8 (low 4 bits) and that + 8 (high 4
    bits); token t at byte 4 (t // 4) + (0, 2, 1, 3)[t % 4]."""
    NP, H, D2, T = v.shape
    t = np.arange(T)
    byt = v[..., 4 * (t // 4) + np.array([0, 2, 1, 3])[t % 4]].astype(np.int64)  # [.., p, t]
    lo, hi = byt & 15, byt >> 4
    out = np.empty((NP, H, 2 * D2, T), np.int64)
    p = np.arange(D2)
    d0 = 16 * (p // 8) + p % 8
    out[:, :, d0, :] = lo
    out[:, :, d0 + 8, :] = hi
    return np.where(out >= 8, out - 16, out)


def stored_codes(cache: HostCache):
    """K [NP,Hkv,P,D] and V [NP,Hkv,D,P] element arrays as stored (codes for FP8/INT4
    decoded to their E4M3 values / integers, before the per-token scale)."""
    if cache.kv_dtype == FP8:
        return e4m3_decode_torch(cache.k), e4m3_decode_torch(cache.v)
    if cache.kv_dtype == INT4:
        return int4_codes(cache.k), int4_v_codes(cache.v)
    if cache.kv_dtype == INT8:  # offset binary: the byte holds code + 128
        return cache.k.astype(np.int64) - 128, cache.v.astype(np.int64) - 128
    return cache.k, cache.v


def logical_kv(cache: HostCache, bt_row, L, g):
    """Reassemble logical K/V [L, D] (float64, dequantised) from the documented layout."""
    t = np.arange(L)
    pages, offs = bt_row[t // P], t % P
    D = cache.head_dim
    dd = np.arange(D)[None, :]
    ks, vs = stored_codes(cache)
    kf = ks.reshape(cache.num_pages, cache.num_kv_heads, -1)
    vf = vs.reshape(cache.num_pages, cache.num_kv_heads, -1)
    k = kf[pages[:, None], g, k_elem(cache.kv_dtype, offs[:, None], dd, D)]
    v = vf[pages[:, None], g, v_elem(cache.kv_dtype, offs[:, None], dd, D)]
    if cache.kv_dtype == BF16:
        k, v = bf16_to_f32(k), bf16_to_f32(v)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    if cache.kv_dtype in QUANTISED:
        k = k * cache.k_scale[pages, g, offs].astype(np.float64)[:, None]
        v = v * cache.v_scale[pages, g, offs].astype(np.float64)[:, None]
    return k, v


def q_f64(q, q_dtype):
    return (bf16_to_f32(q) if q_dtype == BF16 else np.asarray(q, np.float32)).astype(np.float64)


def sdpa(q, k, v, scale, mask=None):
    """torch SDPA in float64: q [n, D], k/v [L, D]."""
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m,
                                                            scale=scale)[0, 0].numpy()


def decode_bruteforce(cache, batch, Hq, Hkv, scale):
    G = Hq // Hkv
    q = q_f64(batch.q, batch.q_dtype)
    out = np.zeros_like(q)
    for b in range(batch.num_seqs):
        L = int(batch.context_lens[b])
        for g in range(Hkv):
            k, v = logical_kv(cache, batch.block_tables[b], L, g)
            out[b, g * G:(g + 1) * G] = sdpa(q[b, g * G:(g + 1) * G], k, v, scale)
    return out


def prefill_bruteforce(cache, batch, Hq, Hkv, scale):
    G = Hq // Hkv
    q = q_f64(batch.q, batch.q_dtype)
    out = np.zeros_like(q)
    for b in range(batch.num_seqs):
        L = int(batch.context_lens[b])
        q0, q1 = int(batch.q_start_loc[b]), int(batch.q_start_loc[b + 1])
        Lq = q1 - q0
        pos = L - Lq + np.arange(Lq)
        mask = np.arange(L)[None, :] <= pos[:, None]
        for g in range(Hkv):
            k, v = logical_kv(cache, batch.block_tables[b], L, g)
            for hh in range(G):
                h = g * G + hh
                out[q0:q1, h] = sdpa(q[q0:q1, h], k, v, scale, mask)
    return out


def run_decode(cache, wl, batch):
    return oracle.decode(cache, batch.q, batch.q_dtype, batch.block_tables,
                         batch.context_lens, wl.scale)


def run_prefill(cache, wl, batch):
    return oracle.prefill(cache, batch.q, batch.q_dtype, batch.q_start_loc,
                          batch.block_tables, batch.context_lens, wl.scale)


# --------------------------------------------------------------------------- BF16 rounding

def check_bf16_rounding():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(500) * 1e30).astype(np.float32),
        (rng.standard_normal(500) * 1e-38).astype(np.float32),  # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], np.float32),
    ])
    # constructed ties: lower 16 bits exactly 0x8000, with even and odd upper halves
    ties = ((rng.integers(0x0080, 0x7f00, 400).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return np.array_equal(ours, ref)


def test_bf16_rounding_matches_library_cast():
    assert check_bf16_rounding()


# --------------------------------------------------------------------------- INT8 quantiser

def check_quantiser():
    rng = np.random.default_rng(11)
    cand = np.arange(-127, 128, dtype=np.float64)
    for trial in range(200):
        n = 64 if trial % 2 == 0 else 128
        x = (rng.standard_normal(n) * (10.0 ** rng.uniform(-3, 3))).astype(np.float32)
        codes, s = oracle.quantize_row_int8(x)
        amax = np.max(np.abs(x))
        if s != np.float32(amax) / np.float32(127.0):
            return False
        if np.any(np.abs(codes.astype(np.int32)) > 127):
            return False
        if np.abs(codes[np.argmax(np.abs(x))]) != 127:
            return False
        # exhaustive nearest code: the chosen code must be (one of) the closest
        r = x.astype(np.float64) / np.float64(s)
        dist = np.abs(r[:, None] - cand[None, :])
        best = dist.min(axis=1)
        mine = np.abs(r - codes.astype(np.float64))
        if np.any(mine > best + 1e-5):
            return False
        # round-trip bound
        if np.any(np.abs(x - codes.astype(np.float64) * s) > 0.5 * s * (1 + 1e-5)):
            return False
    # hand-made ties with s == 1 exactly (max|x| = 127): halves go to the even code
    x = np.zeros(64, np.float32)
    x[0] = 127.0
    x[1:7] = [2.5, 3.5, -2.5, -3.5, 0.5, -0.5]
    codes, s = oracle.quantize_row_int8(x)
    if s != 1.0 or list(codes[:7]) != [127, 2, 4, -2, -4, 0, 0]:
        return False
    # all-zero row
    codes, s = oracle.quantize_row_int8(np.zeros(64, np.float32))
    return s == 0.0 and not codes.any()


def test_int8_quantiser_nearest_code_and_ties():
    assert check_quantiser()


# --------------------------------------------------------------------------- FP8 / INT4

def check_e4m3():
    """The E4M3 decoder against the library's float8 type for all 256 codes, and the
    encoder against the library cast on random values, every tie and the subnormals."""
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_value(codes), e4m3_decode_torch(codes)
    nan = np.isnan(ref)
    if not (np.array_equal(np.isnan(ours), nan) and np.array_equal(ours[~nan], ref[~nan])):
        return False
    rng = np.random.default_rng(21)
    fin = np.array([oracle.e4m3_value(c)[0] for c in range(127)])
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)  # exact ties
    x = np.concatenate([
        (rng.standard_normal(3000) * 10.0 ** rng.uniform(-4, 2.3, 3000)).astype(np.float32),
        mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(500)),
        (rng.uniform(0, 2.0 ** -6, 300)).astype(np.float32),  # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -(2.0 ** -10)], np.float32),
    ])
    x = x[np.abs(x) <= 448]
    if not np.array_equal(oracle.f32_to_e4m3(x), e4m3_torch(x)):
        return False
    # saturation beyond the largest finite value (the encoder's choice; the library cast
    # gives NaN there)
    return list(oracle.f32_to_e4m3([449.0, 1e6, -3e4])) == [0x7E, 0x7E, 0xFE]


def test_e4m3_codec_matches_library_float8():
    assert check_e4m3()


def check_quantisers_fp8_int4():
    rng = np.random.default_rng(13)
    cand = np.arange(-7, 8, dtype=np.float64)
    for trial in range(200):
        n = 64 if trial % 2 == 0 else 128
        x = (rng.standard_normal(n) * (10.0 ** rng.uniform(-3, 3))).astype(np.float32)
        amax = np.max(np.abs(x))
        c4, s4 = oracle.quantize_row_int4(x)
        if s4 != np.float32(amax) / np.float32(7.0) or np.abs(c4[np.argmax(np.abs(x))]) != 7:
            return False
        r = x.astype(np.float64) / np.float64(s4)
        best = np.abs(r[:, None] - cand[None, :]).min(axis=1)
        if np.any(np.abs(r - c4) > best + 1e-5) or np.any(np.abs(c4) > 7):
            return False
        c8, s8 = oracle.quantize_row_fp8(x)
        if s8 != np.float32(amax) / np.float32(448.0):
            return False
        q = np.clip(x / s8, np.float32(-448), np.float32(448))  # float32 division
        if not np.array_equal(c8, e4m3_torch(q)):
            return False
    x = np.zeros(64, np.float32)
    x[:7] = [7.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5]  # s = 1: halves go to the even code
    c4, s4 = oracle.quantize_row_int4(x)
    if s4 != 1.0 or list(c4[:7]) != [7, 2, 4, -2, 0, 0, 2]:
        return False
    c4, s4 = oracle.quantize_row_int4(np.zeros(64, np.float32))
    c8, s8 = oracle.quantize_row_fp8(np.zeros(64, np.float32))
    return s4 == 0 and s8 == 0 and not c4.any() and not c8.any()


def test_fp8_int4_quantisers():
    assert check_quantisers_fp8_int4()


def test_append_fp8_int4_stored_values():
    """Stored codes and scales of every appended row, read back through the documented
    layout (INT4: two codes per byte, the other element of each byte untouched)."""
    for kv in (FP8, INT4):
        wl = W.small_workload(7 + kv, num_q_heads=2, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                              q_dtype=F32, decode_lens=[33, 20])
        c = oracle.cache_from_workload(wl)
        qz = oracle.quantize_row_fp8 if kv == FP8 else oracle.quantize_row_int4
        if kv == FP8:
            ks, vs = c.k, c.v
        else:
            ks, vs = int4_codes(c.k), int4_v_codes(c.v)
        for i in range(wl.slots.shape[0]):
            pg, off = divmod(int(wl.slots[i]), P)
            for h in range(2):
                codes, s = qz(wl.k_src[i, h])
                assert np.array_equal(ks[pg, h, off], codes) and c.k_scale[pg, h, off] == s
                codes, s = qz(wl.v_src[i, h])
                assert np.array_equal(vs[pg, h, :, off], codes) and c.v_scale[pg, h, off] == s


# --------------------------------------------------------------------------- append

def test_append_places_rows_at_documented_positions():
    wl = W.small_workload(5, num_q_heads=4, num_kv_heads=2, head_dim=64, kv_dtype=F32,
                          q_dtype=F32, decode_lens=[20, 37])
    c = HostCache(F32, wl.num_pages, P, 2, 64, fill=np.float32(-7.0))
    rows = np.arange(wl.slots.shape[0])
    sm = wl.slots.copy()
    sm[::5] = -1  # padding tokens are skipped
    assert oracle.append(c, wl.k_src, wl.v_src, F32, sm) == 0
    touched = np.zeros((wl.num_pages, P), bool)
    for i in rows:
        if sm[i] < 0:
            continue
        pg, off = divmod(int(sm[i]), P)
        touched[pg, off] = True
        assert np.array_equal(c.k[pg, :, off, :], wl.k_src[i])
        assert np.array_equal(c.v[pg, :, :, off], wl.v_src[i])
    assert np.all(c.k.transpose(0, 2, 1, 3)[~touched] == -7.0)
    assert np.all(c.v.transpose(0, 3, 1, 2)[~touched] == -7.0)
    # out-of-range slot is reported and skipped
    bad = np.array([wl.num_pages * P + 3], np.int32)
    assert oracle.append(c, wl.k_src[:1], wl.v_src[:1], F32, bad) == 1


def test_append_bf16_and_int8_stored_values():
    wl = W.small_workload(6, num_q_heads=2, num_kv_heads=2, head_dim=64, kv_dtype=INT8,
                          q_dtype=F32, new_dtype=F32, decode_lens=[33])
    ci = oracle.cache_from_workload(wl)
    cb = HostCache(BF16, wl.num_pages, P, 2, 64)
    oracle.append(cb, wl.k_src, wl.v_src, F32, wl.slots)
    for i in range(wl.slots.shape[0]):
        pg, off = divmod(int(wl.slots[i]), P)
        for h in range(2):
            # INT8 bytes hold code + 128 (offset binary)
            codes, s = oracle.quantize_row_int8(wl.k_src[i, h])
            assert np.array_equal(ci.k[pg, h, off].astype(np.int64) - 128, codes)
            assert ci.k_scale[pg, h, off] == s
            codes, s = oracle.quantize_row_int8(wl.v_src[i, h])
            assert np.array_equal(ci.v[pg, h, :, off].astype(np.int64) - 128, codes)
            assert ci.v_scale[pg, h, off] == s
            ref = torch.from_numpy(wl.k_src[i, h]).to(torch.bfloat16).view(torch.int16)
            idx = k_elem(BF16, off, np.arange(64), 64)
            assert np.array_equal(cb.k.reshape(wl.num_pages, 2, -1)[pg, h, idx],
                                  ref.numpy().view(np.uint16))
            ref = torch.from_numpy(wl.v_src[i, h]).to(torch.bfloat16).view(torch.int16)
            idx = v_elem(BF16, off, np.arange(64), 64)
            assert np.array_equal(cb.v.reshape(wl.num_pages, 2, -1)[pg, h, idx],
                                  ref.numpy().view(np.uint16))


# --------------------------------------------------------------------------- dense brute force

CASES = [
    # (kv_dtype, q_dtype, Hq, Hkv, D, decode lens)
    (F32, F32, 9, 3, 64, [1, 15, 16, 17, 37, 64]),
    (BF16, BF16, 12, 2, 128, [5, 31, 32, 33, 70]),
    (BF16, F32, 8, 8, 64, [3, 48]),
    (INT8, F32, 32, 4, 64, [2, 16, 40]),
    (INT8, BF16, 6, 1, 128, [19, 50]),
    (FP8, F32, 8, 2, 64, [1, 17, 40]),
    (FP8, BF16, 6, 1, 128, [19, 33]),
    (INT4, F32, 32, 4, 64, [2, 16, 41]),
    (INT4, BF16, 6, 1, 128, [18, 50]),
]


def check_decode_bruteforce():
    for i, (kv, qd, Hq, Hkv, D, lens) in enumerate(CASES):
        wl = W.small_workload(100 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, decode_lens=lens)
        c = oracle.cache_from_workload(wl)
        bt = wl.batches[0]
        got = run_decode(c, wl, bt)
        ref = decode_bruteforce(c, bt, Hq, Hkv, wl.scale)
        if not np.max(np.abs(got - ref)) <= 1e-12:
            return False
    return True


def test_decode_matches_dense_sdpa():
    assert check_decode_bruteforce()


def check_prefill_bruteforce():
    for i, (kv, qd, Hq, Hkv, D) in enumerate([(BF16, BF16, 12, 2, 128), (F32, F32, 4, 2, 64),
                                              (INT8, F32, 8, 2, 64), (FP8, F32, 8, 2, 64),
                                              (INT4, BF16, 4, 1, 128)]):
        wl = W.small_workload(200 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, prefill=[(20, 13), (0, 17), (33, 1)])
        c = oracle.cache_from_workload(wl)
        bt = wl.batches[0]
        got = run_prefill(c, wl, bt)
        ref = prefill_bruteforce(c, bt, Hq, Hkv, wl.scale)
        if not np.max(np.abs(got - ref)) <= 1e-12:
            return False
    return True


def test_prefill_matches_dense_causal_sdpa():
    assert check_prefill_bruteforce()


# --------------------------------------------------------------------------- closed forms

def _single_seq_cache(D, L, k_rows, v_rows, kv_dtype=F32, Hkv=1):
    npages = (L + P - 1) // P + 2
    c = HostCache(kv_dtype, npages, P, Hkv, D)
    perm = np.random.default_rng(L).permutation(npages).astype(np.int32)
    bt = perm[:(L + P - 1) // P][None, :]
    t = np.arange(L)
    slots = (bt[0, t // P] * P + t % P).astype(np.int32)
    oracle.append(c, k_rows, v_rows, F32, slots)
    return c, bt


def check_closed_forms():
    rng = np.random.default_rng(3)
    D, L = 64, 45
    k = rng.standard_normal((L, 1, D)).astype(np.float32)
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    lens = np.array([L], np.int32)
    # uniform V: output equals that V row
    vrow = rng.standard_normal(D).astype(np.float32)
    c, bt = _single_seq_cache(D, L, k, np.broadcast_to(vrow, (L, 1, D)).copy())
    out = oracle.decode(c, q, F32, bt, lens, 0.125)
    if np.max(np.abs(out[0, 0] - vrow)) > 1e-12:
        return False
    # single token: output equals V_0
    v = rng.standard_normal((L, 1, D)).astype(np.float32)
    c, bt = _single_seq_cache(D, L, k, v)
    out = oracle.decode(c, q, F32, bt, np.array([1], np.int32), 0.125)
    if np.max(np.abs(out[0, 0] - v[0, 0])) > 1e-12:
        return False
    # q = 0: uniform weights, output equals the mean of V
    out = oracle.decode(c, np.zeros_like(q), F32, bt, lens, 0.125)
    if np.max(np.abs(out[0, 0] - v[:, 0].astype(np.float64).mean(axis=0))) > 1e-12:
        return False
    # one key dominating by far more than the exp range: output equals its V row
    kd = np.zeros((L, 1, D), np.float32)
    kd[29, 0, 0] = 1.0e4
    qd = np.zeros((1, 1, D), np.float32)
    qd[0, 0, 0] = 1.0e4
    c, bt = _single_seq_cache(D, L, kd, v)
    out = oracle.decode(c, qd, F32, bt, lens, 1.0)  # score gap 1e8 >> 700 ln 2
    return bool(np.max(np.abs(out[0, 0] - v[29, 0])) <= 1e-12)


def test_closed_forms():
    assert check_closed_forms()


# --------------------------------------------------------------------------- structure

def check_page_permutation_invariance():
    wl = W.small_workload(300, num_q_heads=6, num_kv_heads=2, head_dim=64, kv_dtype=INT8,
                          q_dtype=F32, decode_lens=[50, 17, 64])
    c1 = oracle.cache_from_workload(wl)
    b1 = wl.batches[0]
    out1 = run_decode(c1, wl, b1)
    # remap every page through a fixed permutation and rebuild
    rng = np.random.default_rng(1)
    sigma = rng.permutation(wl.num_pages).astype(np.int32)
    bt2 = np.where(b1.block_tables >= 0, sigma[np.maximum(b1.block_tables, 0)], -1)
    slots2 = (sigma[wl.slots // P] * P + wl.slots % P).astype(np.int32)
    c2 = HostCache(INT8, wl.num_pages, P, 2, 64)
    oracle.append(c2, wl.k_src, wl.v_src, F32, slots2)
    out2 = oracle.decode(c2, b1.q, F32, bt2, b1.context_lens, wl.scale)
    return np.array_equal(out1, out2)


def test_page_permutation_invariance_bit_identical():
    assert check_page_permutation_invariance()


def check_gqa_equals_replicated_mha():
    Hq, Hkv, D = 8, 2, 64
    G = Hq // Hkv
    wl = W.small_workload(301, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, kv_dtype=F32,
                          q_dtype=F32, decode_lens=[23, 40])
    c = oracle.cache_from_workload(wl)
    b = wl.batches[0]
    out = run_decode(c, wl, b)
    mha = HostCache(F32, wl.num_pages, P, Hq, D)
    oracle.append(mha, np.repeat(wl.k_src, G, axis=1), np.repeat(wl.v_src, G, axis=1), F32,
                  wl.slots)
    out2 = oracle.decode(mha, b.q, F32, b.block_tables, b.context_lens, wl.scale)
    return np.array_equal(out, out2)


def test_gqa_equals_mha_with_replicated_kv():
    assert check_gqa_equals_replicated_mha()


def check_causality():
    Hq, Hkv, D = 4, 2, 64
    wl = W.small_workload(302, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, kv_dtype=BF16,
                          q_dtype=BF16, prefill=[(19, 14)])
    c = oracle.cache_from_workload(wl)
    b = wl.batches[0]
    out = run_prefill(c, wl, b)
    L, Lq = 33, 14
    # perturb the K/V of logical positions > p_i for i = 5 -> row 5 unchanged, row 13 changed
    i = 5
    pos = L - Lq + i
    k2 = wl.k_src.copy()
    v2 = wl.v_src.copy()
    k2[pos + 1:] ^= np.uint16(0x1234)
    v2[pos + 1:] ^= np.uint16(0x0f0f)
    c2 = HostCache(BF16, wl.num_pages, P, Hkv, D)
    oracle.append(c2, k2, v2, BF16, wl.slots)
    out2 = run_prefill(c2, wl, b)
    if not np.array_equal(out[:i + 1], out2[:i + 1]) or np.array_equal(out[Lq - 1], out2[Lq - 1]):
        return False
    # the last chunk row equals decode at context L
    dec = oracle.decode(c, b.q[Lq - 1:Lq], BF16, b.block_tables, b.context_lens, wl.scale)
    if not np.array_equal(dec[0], out[Lq - 1]):
        return False
    # every chunk row equals decode with context p_i + 1
    for r in range(Lq):
        d = oracle.decode(c, b.q[r:r + 1], BF16, b.block_tables,
                          np.array([L - Lq + r + 1], np.int32), wl.scale)
        if not np.array_equal(d[0], out[r]):
            return False
    return True


def test_causality_and_prefill_decode_agreement():
    assert check_causality()


def test_invalid_inputs_give_nan_rows_and_counts():
    wl = W.small_workload(303, num_q_heads=2, num_kv_heads=1, head_dim=64, kv_dtype=F32,
                          q_dtype=F32, decode_lens=[20, 20, 0])
    c = oracle.cache_from_workload(wl)
    b = wl.batches[0]
    bt = b.block_tables.copy()
    bt[1, 1] = wl.num_pages + 5
    out = oracle.decode(c, b.q, F32, bt, b.context_lens, wl.scale)
    assert oracle.decode.last_bad == 1
    assert np.all(np.isfinite(out[0])) and np.all(np.isnan(out[1])) and np.all(out[2] == 0)
    lens = b.context_lens.copy()
    lens[0] = bt.shape[1] * P + 1
    out = oracle.decode(c, b.q, F32, b.block_tables, lens, wl.scale)
    assert oracle.decode.last_bad == 1 and np.all(np.isnan(out[0]))


# --------------------------------------------------------------------------- planted mistakes

# --------------------------------------------------------------------------- rotary embedding
# "tinyloop Current Status", model architecture support table (RoPE, configurable theta);
# the half-split pairing (i, i + D/2) is the reading taken.

def rope_complex(x, pos, theta):
    """The rotation written as complex multiplication: pair (x_i, x_{i+D/2}) is the
    complex number x_i + 1j x_{i+D/2}, multiplied by exp(1j * pos * theta^(-2i/D))."""
    x = np.asarray(x, np.float64)
    D = x.shape[0]
    h = D // 2
    z = (x[:h] + 1j * x[h:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(h) / D))
    return np.concatenate([z.real, z.imag])


def check_rope():
    rng = np.random.default_rng(11)
    for D in (64, 128):
        for pos in (0, 1, 37, 4095, 32767):
            for theta in (10000.0, 1.0e6):
                x = rng.standard_normal(D)
                ref = rope_complex(x, pos, theta)
                if np.max(np.abs(oracle.rope_f64(x, pos, theta) - ref)) > 1e-10 * np.abs(x).max():
                    return False
                xf = x.astype(np.float32)
                reff = rope_complex(xf, pos, theta)
                if np.max(np.abs(oracle.rope_f32(xf, pos, theta) - reff)) > 1e-6 * np.abs(x).max():
                    return False
    x = rng.standard_normal(64).astype(np.float32)
    if not np.array_equal(oracle.rope_f32(x, 0, 1.0e4), x):  # position 0: identity
        return False
    # relative positions: <R(q, m), R(k, n)> depends on m - n only
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    a = oracle.rope_f64(q, 100, 1.0e4) @ oracle.rope_f64(k, 40, 1.0e4)
    b = oracle.rope_f64(q, 1060, 1.0e4) @ oracle.rope_f64(k, 1000, 1.0e4)
    return abs(a - b) <= 1e-9 * (1 + abs(a))


def test_rope_is_the_complex_rotation():
    assert check_rope()


# --------------------------------------------------------------------------- decode step

def step_inputs(wl):
    """The newest token of every decode sequence: its source rows, slot and position."""
    batch = wl.batches[0]
    rows = wl.step_rows[:batch.num_seqs]
    return (wl.k_src[rows], wl.v_src[rows], wl.slots[rows].astype(np.int32),
            (batch.context_lens - 1).astype(np.int32))


def copy_cache(c):
    d = HostCache(c.kv_dtype, c.num_pages, c.page_size, c.num_kv_heads, c.head_dim)
    d.k[...] = c.k
    d.v[...] = c.v
    if c.k_scale is not None:
        d.k_scale[...] = c.k_scale
        d.v_scale[...] = c.v_scale
    return d


def same_cache(a, b):
    ok = np.array_equal(a.k, b.k) and np.array_equal(a.v, b.v)
    if a.k_scale is not None:
        ok = ok and np.array_equal(a.k_scale, b.k_scale) and np.array_equal(a.v_scale, b.v_scale)
    return ok


def rows_f32(x, dtype):
    return bf16_to_f32(x) if dtype == BF16 else np.asarray(x, np.float32)


def check_decode_step():
    theta = 1.0e4
    for i, (kv, qd, Hq, Hkv, D, lens) in enumerate(CASES):
        wl = W.small_workload(400 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, decode_lens=lens)
        batch = wl.batches[0]
        hist = oracle.cache_from_workload(wl, rows=wl.history_rows)
        k_new, v_new, slots, pos = step_inputs(wl)
        args = (batch.block_tables, batch.context_lens, wl.scale)
        # no rotation: exactly append, then decode
        c1, c2 = copy_cache(hist), copy_cache(hist)
        got = oracle.decode_step(c1, batch.q, qd, k_new, v_new, wl.new_dtype, slots, None,
                                 theta, *args)
        oracle.append(c2, k_new, v_new, wl.new_dtype, slots)
        if not (same_cache(c1, c2) and np.array_equal(got, oracle.decode(c2, batch.q, qd, *args))):
            return False
        # rotation: the stored keys are the float-form rotation of the inputs, and the output
        # is dense attention of the double-form rotated queries over the reassembled cache
        c3, c4 = copy_cache(hist), copy_cache(hist)
        got = oracle.decode_step(c3, batch.q, qd, k_new, v_new, wl.new_dtype, slots, pos,
                                 theta, *args)
        kf = rows_f32(k_new, wl.new_dtype)
        krot = np.stack([[oracle.rope_f32(kf[b, h], pos[b], theta) for h in range(Hkv)]
                         for b in range(batch.num_seqs)])
        oracle.append(c4, krot, rows_f32(v_new, wl.new_dtype), F32, slots)
        if not same_cache(c3, c4):
            return False
        G = Hq // Hkv
        q = q_f64(batch.q, qd)
        for b in range(batch.num_seqs):
            L = int(batch.context_lens[b])
            for g in range(Hkv):
                k, v = logical_kv(c4, batch.block_tables[b], L, g)
                qr = np.stack([oracle.rope_f64(q[b, h], pos[b], theta) for h in range(g * G, (g + 1) * G)])
                if np.max(np.abs(got[b, g * G:(g + 1) * G] - sdpa(qr, k, v, wl.scale))) > 1e-12:
                    return False
        # a slot that is not position L - 1's slot: NaN rows, nothing stored
        c5 = copy_cache(hist)
        bad = slots.copy()
        bad[0] = (bad[0] + 1) % (wl.num_pages * P)
        got = oracle.decode_step(c5, batch.q, qd, k_new, v_new, wl.new_dtype, bad, pos, theta,
                                 *args, seqs=[0])
        if not (np.all(np.isnan(got[0])) and oracle.decode_step.last_bad == 1 and same_cache(c5, hist)):
            return False
    return True


def test_decode_step_is_rotate_store_attend():
    assert check_decode_step()


# --------------------------------------------------------------------------- sliding window
# "tinyloop Current Status", KV cache modes table (a cache window bounds KV storage); the
# reading taken: position pos sees positions pos - W + 1 .. pos, pages wholly before that
# are never read.

WINDOW_CASES = [
    # kv, q, Hq, Hkv, D, decode lens, windows
    (F32, F32, 4, 2, 64, [45, 16, 1, 70, 33], [1, 5, 16, 17, 33, 100]),
    (BF16, BF16, 12, 2, 128, [40, 97], [3, 32, 47]),
    (INT8, F32, 8, 2, 64, [50, 18], [2, 16, 31]),
]


def check_window_decode():
    """Decode with a window equals dense attention over the reassembled rows
    max(0, L - W) .. L - 1, whatever the table holds for the pages before them."""
    for i, (kv, qd, Hq, Hkv, D, lens, wins) in enumerate(WINDOW_CASES):
        wl = W.small_workload(500 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, decode_lens=lens)
        c = oracle.cache_from_workload(wl)
        b = wl.batches[0]
        q = q_f64(b.q, qd)
        G = Hq // Hkv
        for win in wins:
            got = oracle.decode(c, b.q, qd, b.block_tables, b.context_lens, wl.scale, window=win)
            for s in range(b.num_seqs):
                L = int(b.context_lens[s])
                lo = max(0, L - win)
                for g in range(Hkv):
                    k, v = logical_kv(c, b.block_tables[s], L, g)
                    ref = sdpa(q[s, g * G:(g + 1) * G], k[lo:], v[lo:], wl.scale)
                    if not np.max(np.abs(got[s, g * G:(g + 1) * G] - ref)) <= 1e-12:
                        return False
            # pages wholly before the window released (-1): same result, no error
            bt = b.block_tables.copy()
            for s in range(b.num_seqs):
                bt[s, :max(0, int(b.context_lens[s]) - win) // P] = -1
            got2 = oracle.decode(c, b.q, qd, bt, b.context_lens, wl.scale, window=win)
            if oracle.decode.last_bad != 0 or not np.array_equal(got, got2):
                return False
    # window 1: the output is the newest V row itself (FP32 cache stores rows exactly)
    wl = W.small_workload(510, num_q_heads=6, num_kv_heads=3, head_dim=64, kv_dtype=F32,
                          q_dtype=F32, decode_lens=[29, 1, 48])
    c = oracle.cache_from_workload(wl)
    b = wl.batches[0]
    got = oracle.decode(c, b.q, F32, b.block_tables, b.context_lens, wl.scale, window=1)
    newest = wl.v_src[wl.step_rows[:3]].astype(np.float64)  # [B, Hkv, D]
    if not np.array_equal(got, np.repeat(newest, 2, axis=1)):
        return False
    # a window at least as long as every context is plain causal attention
    full = oracle.decode(c, b.q, F32, b.block_tables, b.context_lens, wl.scale)
    return np.array_equal(full, oracle.decode(c, b.q, F32, b.block_tables, b.context_lens,
                                              wl.scale, window=48))


def test_window_decode_is_attention_over_the_last_w():
    assert check_window_decode()


def check_window_prefill():
    """Each chunk row sees max(0, pos - W + 1) .. pos: dense attention with a band mask."""
    for i, (kv, qd, Hq, Hkv, D) in enumerate([(BF16, BF16, 12, 2, 128), (F32, F32, 4, 2, 64),
                                              (INT8, F32, 8, 2, 64)]):
        wl = W.small_workload(520 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, prefill=[(20, 13), (0, 17), (33, 1),
                                                                (5, 40)])
        c = oracle.cache_from_workload(wl)
        b = wl.batches[0]
        q = q_f64(b.q, qd)
        G = Hq // Hkv
        for win in (1, 7, 16, 30):
            got = oracle.prefill(c, b.q, qd, b.q_start_loc, b.block_tables, b.context_lens,
                                 wl.scale, window=win)
            for s in range(b.num_seqs):
                L = int(b.context_lens[s])
                q0, q1 = int(b.q_start_loc[s]), int(b.q_start_loc[s + 1])
                pos = L - (q1 - q0) + np.arange(q1 - q0)
                t = np.arange(L)[None, :]
                mask = (t <= pos[:, None]) & (t > pos[:, None] - win)
                for g in range(Hkv):
                    k, v = logical_kv(c, b.block_tables[s], L, g)
                    for h in range(g * G, (g + 1) * G):
                        ref = sdpa(q[q0:q1, h], k, v, wl.scale, mask)
                        if not np.max(np.abs(got[q0:q1, h] - ref)) <= 1e-12:
                            return False
    return True


def test_window_prefill_is_banded_causal_attention():
    assert check_window_prefill()


def check_window_step():
    """The decode step with a window is the step's store followed by windowed decode."""
    theta = 1.0e4
    for i, (kv, qd, Hq, Hkv, D, lens, wins) in enumerate(WINDOW_CASES):
        wl = W.small_workload(530 + i, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              kv_dtype=kv, q_dtype=qd, decode_lens=lens)
        b = wl.batches[0]
        hist = oracle.cache_from_workload(wl, rows=wl.history_rows)
        k_new, v_new, slots, pos = step_inputs(wl)
        for win in wins[:2]:
            c1, c2 = copy_cache(hist), copy_cache(hist)
            got = oracle.decode_step(c1, b.q, qd, k_new, v_new, wl.new_dtype, slots, None, theta,
                                     b.block_tables, b.context_lens, wl.scale, window=win)
            oracle.append(c2, k_new, v_new, wl.new_dtype, slots)
            ref = oracle.decode(c2, b.q, qd, b.block_tables, b.context_lens, wl.scale, window=win)
            if not (same_cache(c1, c2) and np.array_equal(got, ref)):
                return False
    return True


def test_window_step_is_store_then_windowed_decode():
    assert check_window_step()


PINS = [check_bf16_rounding, check_quantiser, check_decode_bruteforce,
        check_prefill_bruteforce, check_closed_forms, check_page_permutation_invariance,
        check_gqa_equals_replicated_mha, check_causality, check_rope, check_decode_step,
        check_window_decode, check_window_prefill, check_window_step, check_e4m3,
        check_quantisers_fp8_int4]


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16])
def test_planted_mistake_is_caught(mutant, monkeypatch):
    path = oracle.build(defines=[f"ORACLE_MUTANT={mutant}"], name=f"liboracle_m{mutant}.so")
    monkeypatch.setattr(oracle, "_lib", oracle.load(path))
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin()
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


def test_default_build_passes_every_pin():
    for pin in PINS:
        assert pin(), pin.__name__
