"""Seeded synthetic inputs for paged GQA attention.

This module only draws inputs: context lengths, page tables, queries and the source
K/V rows that the append step writes into the cache.  It holds none of the attention
arithmetic, so both the CUDA library's tests and the CPU oracle can take their inputs
from here without sharing any part of the method.

Shapes follow the model families the pages name ("Tiny-LLM-Inference Project_Status":
SmolLM2-135M and Qwen2.5-1.5B; "mini-llm-inference-engine" README: TinyLlama 1.1B) and
the 16-token pages of "tinyloop Current Status", KV cache modes table.  Values are
N(0, 1) from a CPU ``torch.Generator`` seeded with ``1000 + index``; BF16 data is drawn
in float32 and cast with torch's round-to-nearest-even cast.  Page tables come from one
``torch.randperm`` over the pool, consumed in order, ceil(L/16) pages per sequence;
unused table entries hold -1 and are never read.

No public dataset or trained weight is involved: every value is synthetic.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

F32, BF16, INT8, FP8, INT4 = 0, 1, 2, 3, 4
DTYPE_NAMES = {F32: "f32", BF16: "bf16", INT8: "int8", FP8: "fp8", INT4: "int4"}
PAGE_SIZE = 16


@dataclasses.dataclass
class Batch:
    """One batch of sequences over one page pool.

    ``kind`` is "decode" (one query token per sequence) or "prefill" (a causal chunk of
    ``chunk_lens[b]`` query tokens at the end of each sequence's context).
    Arrays are numpy; BF16 arrays hold raw bfloat16 bit patterns as uint16.
    """

    kind: str
    context_lens: np.ndarray  # int32 [B]   tokens in cache after this step's append
    block_tables: np.ndarray  # int32 [B, MB]
    q: np.ndarray  # [B, Hq, D] (decode) or [sum Lq, Hq, D] (prefill); f32 or bf16 bits
    q_dtype: int
    chunk_lens: Optional[np.ndarray] = None  # int32 [B] (prefill only)
    q_start_loc: Optional[np.ndarray] = None  # int32 [B+1] (prefill only)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    kv_dtype: int
    new_dtype: int  # dtype of the source K/V rows handed to append
    scale: float
    batches: list  # list[Batch]
    # Source rows of every cached token, in append order, and their slots.
    k_src: np.ndarray  # [T, Hkv, D] f32 or bf16 bits
    v_src: np.ndarray
    slots: np.ndarray  # int32 [T]
    # Which of the T source rows are written inside the timed step (the newest token of
    # every decode sequence and the whole chunk of every prefill sequence); the rest
    # are the "history" already in cache when the step starts.
    step_rows: np.ndarray  # int64 indices into [T]

    @property
    def history_rows(self) -> np.ndarray:
        mask = np.ones(self.slots.shape[0], dtype=bool)
        mask[self.step_rows] = False
        return np.nonzero(mask)[0]


def _randn(g: torch.Generator, shape, dtype: int) -> np.ndarray:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if dtype == BF16:
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    return x.numpy().copy()


def _pages_for(lens, P):
    return [int(math.ceil(int(L) / P)) for L in lens]


def make_workload(
    name: str,
    *,
    seed: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    num_pages: int,
    kv_dtype: int,
    q_dtype: int,
    new_dtype: int,
    decode_lens=(),
    max_decode_len: Optional[int] = None,
    prefill=(),  # sequence of (prior_len, chunk_len)
    max_prefill_len: Optional[int] = None,
    page_size: int = PAGE_SIZE,
    scale: Optional[float] = None,
) -> Workload:
    """Draw a workload deterministically from ``seed``.

    Draw order (fixed): page permutation, decode queries, prefill queries, then K and V
    source rows sequence by sequence (decode sequences first) in logical token order.
    """
    g = torch.Generator().manual_seed(seed)
    P, Hq, Hkv, D = page_size, num_q_heads, num_kv_heads, head_dim
    decode_lens = [int(x) for x in decode_lens]
    prefill = [(int(a), int(c)) for a, c in prefill]
    pre_lens = [a + c for a, c in prefill]
    need = sum(_pages_for(decode_lens, P)) + sum(_pages_for(pre_lens, P))
    if need > num_pages:
        raise ValueError(f"{name}: {need} pages needed, pool has {num_pages}")
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    cursor = 0

    def tables(lens, max_len):
        nonlocal cursor
        mb = max(1, int(math.ceil((max_len if max_len else max(lens or [1])) / P)))
        bt = np.full((len(lens), mb), -1, dtype=np.int32)
        for b, L in enumerate(lens):
            n = int(math.ceil(L / P))
            bt[b, :n] = perm[cursor:cursor + n]
            cursor += n
        return bt

    dec_bt = tables(decode_lens, max_decode_len) if decode_lens else None
    pre_bt = tables(pre_lens, max_prefill_len) if prefill else None

    batches = []
    if decode_lens:
        q = _randn(g, (len(decode_lens), Hq, D), q_dtype)
        batches.append(Batch("decode", np.array(decode_lens, np.int32), dec_bt, q, q_dtype))
    if prefill:
        chunk = np.array([c for _, c in prefill], np.int32)
        qsl = np.zeros(len(prefill) + 1, np.int32)
        qsl[1:] = np.cumsum(chunk)
        q = _randn(g, (int(qsl[-1]), Hq, D), q_dtype)
        batches.append(Batch("prefill", np.array(pre_lens, np.int32), pre_bt, q, q_dtype,
                             chunk_lens=chunk, q_start_loc=qsl))

    # Source rows in logical order; the step rows are the last token of each decode
    # sequence and the chunk of each prefill sequence.
    slots, step = [], []
    row = 0
    for lens, bt, chunks in ((decode_lens, dec_bt, [1] * len(decode_lens)),
                             (pre_lens, pre_bt, [c for _, c in prefill])):
        for b, L in enumerate(lens):
            t = np.arange(L, dtype=np.int64)
            slots.append(bt[b, t // P].astype(np.int64) * P + t % P)
            step.append(row + np.arange(L - chunks[b], L, dtype=np.int64))
            row += L
    slots = np.concatenate(slots).astype(np.int32) if slots else np.zeros(0, np.int32)
    step = np.concatenate(step) if step else np.zeros(0, np.int64)
    T = int(slots.shape[0])
    k_src = _randn(g, (T, Hkv, D), new_dtype)
    v_src = _randn(g, (T, Hkv, D), new_dtype)
    return Workload(name, Hq, Hkv, D, P, num_pages, kv_dtype, new_dtype,
                    float(scale if scale is not None else 1.0 / math.sqrt(D)),
                    batches, k_src, v_src, slots, step)


def _uniform_lens(seed: int, n: int, lo: int, hi: int):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# The named workloads.  Index i uses seed 1000 + i (lengths use 2000 + i).  The last two
# are the batch-256 TinyLlama-shaped decode with the cache in FP8 and in INT4.
WORKLOADS = ("tiny", "smollm2-f32", "qwen-bf16", "tinyllama-int8", "mixed", "tinyllama-fp8",
             "tinyllama-int4")


def workload(name: str) -> Workload:
    if name == "tiny":
        # batch 1, 9 Q / 3 KV heads, head_dim 64, 37 cached tokens (last page partial),
        # FP32 everywhere, a pool of 8 pages in random order.
        return make_workload(name, seed=1000, num_q_heads=9, num_kv_heads=3, head_dim=64,
                             num_pages=8, kv_dtype=F32, q_dtype=F32, new_dtype=F32,
                             decode_lens=[37], max_decode_len=37)
    if name == "smollm2-f32":
        lens = _uniform_lens(2001, 64, 128, 1024)
        return make_workload(name, seed=1001, num_q_heads=9, num_kv_heads=3, head_dim=64,
                             num_pages=4096, kv_dtype=F32, q_dtype=F32, new_dtype=F32,
                             decode_lens=lens, max_decode_len=1024)
    if name == "qwen-bf16":
        lens = _uniform_lens(2002, 32, 512, 4096)
        return make_workload(name, seed=1002, num_q_heads=12, num_kv_heads=2, head_dim=128,
                             num_pages=16384, kv_dtype=BF16, q_dtype=BF16, new_dtype=BF16,
                             decode_lens=lens, max_decode_len=4096)
    if name == "tinyllama-int8":
        return make_workload(name, seed=1003, num_q_heads=32, num_kv_heads=4, head_dim=64,
                             num_pages=16384, kv_dtype=INT8, q_dtype=F32, new_dtype=F32,
                             decode_lens=[1024] * 256, max_decode_len=1024)
    if name in ("tinyllama-fp8", "tinyllama-int4"):
        fp8 = name == "tinyllama-fp8"
        return make_workload(name, seed=1005 if fp8 else 1006, num_q_heads=32, num_kv_heads=4,
                             head_dim=64, num_pages=16384, kv_dtype=FP8 if fp8 else INT4,
                             q_dtype=F32, new_dtype=F32, decode_lens=[1024] * 256,
                             max_decode_len=1024)
    if name == "mixed":
        return make_workload(name, seed=1004, num_q_heads=12, num_kv_heads=2, head_dim=128,
                             num_pages=16384, kv_dtype=BF16, q_dtype=BF16, new_dtype=BF16,
                             decode_lens=[32768] * 4, max_decode_len=32768,
                             prefill=[(2048, 512)] * 2, max_prefill_len=2560)
    raise KeyError(name)


def small_workload(seed: int, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   kv_dtype: int, q_dtype: int, new_dtype: Optional[int] = None,
                   decode_lens=(), prefill=(), num_pages: Optional[int] = None,
                   max_decode_len=None, max_prefill_len=None, scale=None) -> Workload:
    """A parity-sized workload (the oracle finishes it in well under a second)."""
    P = PAGE_SIZE
    need = sum(_pages_for(decode_lens, P)) + sum(_pages_for([a + c for a, c in prefill], P))
    if num_pages is None:
        num_pages = max(4, need + 3)
    if new_dtype is None:
        new_dtype = BF16 if kv_dtype == BF16 else F32
    return make_workload(f"small-{seed}", seed=seed, num_q_heads=num_q_heads,
                         num_kv_heads=num_kv_heads, head_dim=head_dim, num_pages=num_pages,
                         kv_dtype=kv_dtype, q_dtype=q_dtype, new_dtype=new_dtype,
                         decode_lens=decode_lens, max_decode_len=max_decode_len,
                         prefill=prefill, max_prefill_len=max_prefill_len, scale=scale)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (a data-format conversion)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def cache_shapes(wl: Workload):
    """Physical cache shapes: K [NP, Hkv, P, D], V [NP, Hkv, D, P], scales [NP, Hkv, P]."""
    NP, H, P, D = wl.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim
    return (NP, H, P, D), (NP, H, D, P), (NP, H, P)
