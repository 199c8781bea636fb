"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

TOL = {W.F32: 1e-4, W.BF16: 2e-3, W.INT8: 2e-3, W.FP8: 2e-3, W.INT4: 2e-3}


def oracle_outputs(wl, oc=None, seqs=None):
    oc = oc if oc is not None else oracle.cache_from_workload(wl)
    outs = []
    for b in wl.batches:
        if b.kind == "decode":
            outs.append(oracle.decode(oc, b.q, b.q_dtype, b.block_tables, b.context_lens,
                                      wl.scale, seqs=seqs))
        else:
            outs.append(oracle.prefill(oc, b.q, b.q_dtype, b.q_start_loc, b.block_tables,
                                       b.context_lens, wl.scale, seqs=seqs))
    return outs


def gpu_outputs(wl, cache_fill=None, chunk_pages=0, key_split=0):
    """One step of the workload through the library (chunk_pages: the decode calls'
    split-K pages per block, 0 = automatic; key_split: the prefill calls' option);
    outputs, device status, device workload."""
    dw = runner.upload(wl, "cuda", cache_fill=cache_fill, split_pages=chunk_pages,
                       key_split=key_split)
    outs = runner.run_step(dw)
    torch.cuda.synchronize()
    status = int(dw.dev_status.item())
    return [o.cpu().numpy().astype(np.float64) for o in outs], status, dw


def max_err(a, b, rows=None):
    if rows is not None:
        a, b = a[rows], b[rows]
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def cache_bytes_equal(dw, oc):
    """Compare the GPU cache with the oracle's cache byte for byte."""
    k = dw.cache.k.cpu()
    v = dw.cache.v.cpu()
    if k.dtype == torch.bfloat16:
        k = k.view(torch.int16).numpy().view(np.uint16)
        v = v.view(torch.int16).numpy().view(np.uint16)
    else:
        k, v = k.numpy(), v.numpy()
    ok = np.array_equal(k.view(np.uint8), oc.k.view(np.uint8)) and \
        np.array_equal(v.view(np.uint8), oc.v.view(np.uint8))
    if oc.k_scale is not None:
        ok = ok and np.array_equal(dw.cache.k_scale.cpu().numpy().view(np.uint32),
                                   oc.k_scale.view(np.uint32))
        ok = ok and np.array_equal(dw.cache.v_scale.cpu().numpy().view(np.uint32),
                                   oc.v_scale.view(np.uint32))
    return ok
