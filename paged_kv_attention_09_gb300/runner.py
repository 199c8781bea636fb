"""Drive a synthetic workload through the library on one GPU.

Moves a ``workloads.Workload`` to device tensors, fills its cache through
``pkv_append`` and runs the decode / prefill calls.  Used by the GPU tests, the smoke
check and the benchmark; all arithmetic happens in libpkv's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import pkv
from .workloads import BF16, F32, Workload


def np_to_torch(a: np.ndarray, dtype_code: Optional[int] = None) -> torch.Tensor:
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


@dataclasses.dataclass
class DeviceBatch:
    kind: str
    q: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    q_start_loc: Optional[torch.Tensor]
    max_q_len: int
    out: torch.Tensor
    workspace: Optional[torch.Tensor]


@dataclasses.dataclass
class DeviceWorkload:
    wl: Workload
    cache: pkv.KVCache
    k_src: torch.Tensor
    v_src: torch.Tensor
    slots: torch.Tensor
    step_rows: torch.Tensor
    batches: list
    dev_status: torch.Tensor
    split_pages: int = 0  # decode split-K pages per block (0: automatic)
    key_split: int = 0    # prefill blocks per row tile's keys (0: automatic)


def upload(wl: Workload, device="cuda", cache_fill: Optional[float] = None,
           fill_history: bool = True, split_pages: int = 0,
           key_split: int = 0) -> DeviceWorkload:
    """Allocate the cache and batch tensors; optionally append the history rows.
    ``split_pages``: the decode calls' split-K pages per block (0: automatic);
    ``key_split``: the prefill calls' option (pkv_prefill_opts)."""
    cache = pkv.KVCache.allocate(wl.num_pages, wl.num_kv_heads, wl.head_dim, wl.kv_dtype, device)
    if cache_fill is not None:  # sentinel for never-written slots (NaN poisons padding)
        if wl.kv_dtype in pkv.CODED:
            cache.k_scale.fill_(cache_fill)
            cache.v_scale.fill_(cache_fill)
            if wl.kv_dtype == pkv.FP8 and cache_fill != cache_fill:  # NaN: the E4M3 NaN code
                cache.k.fill_(0x7F)
                cache.v.fill_(0x7F)
        else:
            cache.k.fill_(cache_fill)
            cache.v.fill_(cache_fill)
    k_src = np_to_torch(wl.k_src).to(device)
    v_src = np_to_torch(wl.v_src).to(device)
    slots = torch.from_numpy(wl.slots).to(device)
    step_rows = torch.from_numpy(wl.step_rows).to(device)
    batches = []
    for b in wl.batches:
        q = np_to_torch(b.q).to(device)
        B, Hq, D = b.num_seqs, wl.num_q_heads, wl.head_dim
        qsl = None if b.q_start_loc is None else torch.from_numpy(b.q_start_loc).to(device)
        max_q = int(b.chunk_lens.max()) if b.chunk_lens is not None and len(b.chunk_lens) else 1
        out = torch.empty(q.shape[0], Hq, D, dtype=torch.float32, device=device)
        if b.kind == "decode":
            nbytes = pkv.pkv_decode_workspace_size(cache, B, Hq, b.max_blocks, split_pages)
        else:
            nbytes = pkv.pkv_prefill_workspace_size(cache, B, Hq, max_q, b.max_blocks,
                                                    key_split)
        batches.append(DeviceBatch(b.kind, q, torch.from_numpy(b.block_tables).to(device),
                                   torch.from_numpy(b.context_lens).to(device), qsl, max_q, out,
                                   pkv.workspace_for(nbytes, device)))
    dw = DeviceWorkload(wl, cache, k_src, v_src, slots, step_rows, batches,
                        torch.zeros(1, dtype=torch.int32, device=device), split_pages,
                        key_split)
    if fill_history:
        hist = torch.from_numpy(wl.history_rows).to(device)
        append_rows(dw, hist)
    return dw


def append_rows(dw: DeviceWorkload, rows: torch.Tensor, stream=None) -> None:
    if rows.numel() == 0:
        return
    pkv.pkv_append(dw.cache, dw.k_src[rows].contiguous(), dw.v_src[rows].contiguous(),
                   dw.slots[rows].contiguous(), dw.dev_status, stream)


def run_batch(dw: DeviceWorkload, i: int, stream=None, bound: bool = False):
    """Batch ``i``'s attention; returns its output, or (bound=True) the call itself as a
    pkv.BoundCall, not yet issued."""
    b = dw.batches[i]
    if b.kind == "decode":
        call = pkv.pkv_decode_attn(dw.cache, b.q, b.block_tables, b.context_lens, dw.wl.scale,
                                   b.out, b.workspace, dw.dev_status, stream,
                                   split_pages=dw.split_pages, bound=bound)
    else:
        call = pkv.pkv_prefill_chunk_attn(dw.cache, b.q, b.q_start_loc, b.max_q_len,
                                          b.block_tables, b.context_lens, dw.wl.scale, b.out,
                                          b.workspace, dw.dev_status, stream,
                                          key_split=dw.key_split, bound=bound)
    return call if bound else b.out


def run_step(dw: DeviceWorkload, step_k=None, step_v=None, step_slots=None, stream=None):
    """One pass of the hot path: append the step's new rows, then every batch's attention."""
    if step_k is None:
        rows = dw.step_rows
        step_k, step_v, step_slots = dw.k_src[rows], dw.v_src[rows], dw.slots[rows]
    if step_slots.numel():
        pkv.pkv_append(dw.cache, step_k, step_v, step_slots, dw.dev_status, stream)
    return [run_batch(dw, i, stream) for i in range(len(dw.batches))]


def decode_step_inputs(dw: DeviceWorkload, i: int = 0, rope: bool = True):
    """The new token of every sequence of decode batch ``i`` (the workload's newest row of
    each decode sequence): K and V rows, slots, and rotation positions (context - 1)."""
    b = dw.batches[i]
    B = b.q.shape[0]
    rows = dw.step_rows[:B]
    pos = (b.context_lens - 1).to(torch.int32).contiguous() if rope else None
    return (dw.k_src[rows].contiguous(), dw.v_src[rows].contiguous(),
            dw.slots[rows].contiguous(), pos)


def run_decode_step(dw: DeviceWorkload, inputs, i: int = 0, rope_theta: float = 10000.0,
                    stream=None, bound: bool = False):
    """Decode batch ``i`` as one fused step (rotate, append the new rows, attend); returns
    its output, or (bound=True) the call as a pkv.BoundCall, not yet issued."""
    b = dw.batches[i]
    k, v, slots, pos = inputs
    call = pkv.pkv_decode_step(dw.cache, b.q, k, v, slots, pos, rope_theta, b.block_tables,
                               b.context_lens, dw.wl.scale, b.out, b.workspace, dw.dev_status,
                               stream, split_pages=dw.split_pages, bound=bound)
    return call if bound else b.out
