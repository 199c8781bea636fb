"""CPU oracle for paged GQA attention (FP64) — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision, compiled with
``-ffp-contract=off`` and without fast-math).  This module compiles it on first use and
wraps it with numpy arrays.  Every function states the passage it follows in the C
source; the pins that tie it to something other than itself are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
F32, BF16, INT8, FP8, INT4 = 0, 1, 2, 3, 4
QUANTISED = (INT8, FP8, INT4)


def build(force: bool = False, defines=(), name: str = "liboracle.so") -> str:
    """Compile the oracle into ``oracle/_build/<name>``; returns the path.

    ``defines`` lets the pin tests build deliberately broken variants of the oracle to
    show that the pins catch them.
    """
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, name)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-std=c99", *[f"-D{d}" for d in defines], "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_lib = None
_lock = threading.Lock()


def _bind(lib):
    p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_quantize_row_int8.argtypes = [p, i, p, p]
    lib.oracle_quantize_row_int8.restype = None
    lib.oracle_quantize_row_fp8.argtypes = [p, i, p, p]
    lib.oracle_quantize_row_fp8.restype = None
    lib.oracle_quantize_row_int4.argtypes = [p, i, p, p]
    lib.oracle_quantize_row_int4.restype = None
    lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_append.argtypes = [i, i, i, i, i, p, p, p, p, p, p, i, p, i]
    lib.oracle_append.restype = i
    lib.oracle_decode.argtypes = [i, i, i, i, i, p, p, p, p, p, i, i, i, p, i, p, d, i, p, i, i]
    lib.oracle_decode.restype = i
    lib.oracle_prefill.argtypes = [i, i, i, i, i, p, p, p, p, p, i, i, i, p, p, i, p, d, i, p, i,
                                   i]
    lib.oracle_prefill.restype = i
    lib.oracle_rope_f64.argtypes = [p, p, i, i, d]
    lib.oracle_rope_f64.restype = None
    lib.oracle_rope_f32.argtypes = [p, p, i, i, d]
    lib.oracle_rope_f32.restype = None
    lib.oracle_decode_step.argtypes = [i, i, i, i, i, p, p, p, p, p, i, p, p, i, p, p, d, i, i,
                                       p, i, p, d, i, p, i, i]
    lib.oracle_decode_step.restype = i
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads a specific build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_REAL = {F32: np.float32, BF16: np.uint16}
# element containers: INT8 bytes hold code + 128 (offset binary), FP8 bytes E4M3 codes,
# INT4 bytes two codes each
_CACHE = {F32: np.float32, BF16: np.uint16, INT8: np.uint8, FP8: np.uint8, INT4: np.uint8}


class HostCache:
    """The oracle's own KV cache: K [NP,Hkv,P,D], V [NP,Hkv,D,P], scales [NP,Hkv,P]
    (INT4: K [NP,Hkv,P,D/2] and V [NP,Hkv,D/2,P] bytes, two codes per byte)."""

    def __init__(self, kv_dtype, num_pages, page_size, num_kv_heads, head_dim, fill=0):
        self.kv_dtype, self.num_pages, self.page_size = kv_dtype, num_pages, page_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        NP, H, P, D = num_pages, num_kv_heads, page_size, head_dim
        dt = _CACHE[kv_dtype]
        if kv_dtype == INT4:  # two codes per byte: K rows of D/2, V row pairs of P bytes
            self.k = np.full((NP, H, P, D // 2), fill, dtype=dt)
            self.v = np.full((NP, H, D // 2, P), fill, dtype=dt)
        else:
            self.k = np.full((NP, H, P, D), fill, dtype=dt)
            self.v = np.full((NP, H, D, P), fill, dtype=dt)
        if kv_dtype in QUANTISED:
            self.k_scale = np.zeros((NP, H, P), np.float32)
            self.v_scale = np.zeros((NP, H, P), np.float32)
        else:
            self.k_scale = self.v_scale = None

    def args(self):
        return (self.kv_dtype, self.num_pages, self.page_size, self.num_kv_heads,
                self.head_dim, _ptr(self.k), _ptr(self.v), _ptr(self.k_scale),
                _ptr(self.v_scale))


def f32_to_bf16(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    lib = load()
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in x], np.uint16)


def quantize_row_int8(x):
    """Symmetric INT8 quantisation of one row; returns (codes int8, scale float32)."""
    x = _c(x, np.float32)
    codes = np.zeros(x.shape[0], np.int8)
    s = np.zeros(1, np.float32)
    load().oracle_quantize_row_int8(_ptr(x), x.shape[0], _ptr(codes), _ptr(s))
    return codes, s[0]


def quantize_row_fp8(x):
    """Symmetric FP8 (E4M3) quantisation of one row; returns (codes uint8, scale float32)."""
    x = _c(x, np.float32)
    codes = np.zeros(x.shape[0], np.uint8)
    s = np.zeros(1, np.float32)
    load().oracle_quantize_row_fp8(_ptr(x), x.shape[0], _ptr(codes), _ptr(s))
    return codes, s[0]


def quantize_row_int4(x):
    """Symmetric INT4 quantisation of one row; returns (codes int8 in [-7, 7], scale)."""
    x = _c(x, np.float32)
    codes = np.zeros(x.shape[0], np.int8)
    s = np.zeros(1, np.float32)
    load().oracle_quantize_row_int4(_ptr(x), x.shape[0], _ptr(codes), _ptr(s))
    return codes, s[0]


def f32_to_e4m3(x) -> np.ndarray:
    """Encode float32 values as FP8 E4M3 codes (nearest, ties to even, saturating)."""
    lib = load()
    return np.array([lib.oracle_f32_to_e4m3(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    np.uint8)


def e4m3_value(codes) -> np.ndarray:
    lib = load()
    return np.array([lib.oracle_e4m3_value(int(c)) for c in np.asarray(codes).ravel()])


def append(cache: HostCache, k_new, v_new, new_dtype, slot_mapping) -> int:
    """Write rows [T,Hkv,D] into ``cache`` at ``slot_mapping``; returns #bad slots."""
    k_new = _c(k_new, _REAL[new_dtype])
    v_new = _c(v_new, _REAL[new_dtype])
    sm = _c(slot_mapping, np.int32)
    return load().oracle_append(*cache.args()[:9], _ptr(k_new), _ptr(v_new), new_dtype,
                                _ptr(sm), int(sm.shape[0]))


def _threads(n_items, threads):
    if threads is None:
        threads = 1
    return max(1, min(int(threads), n_items))


def decode(cache: HostCache, q, q_dtype, block_tables, context_lens, scale, *,
           window=0, seqs=None, threads=None):
    """Decode attention in FP64 for every sequence (or the listed ``seqs``).

    ``window`` > 0: each query attends to the last ``window`` positions only.

    Returns float64 [B, Hq, D]; rows of sequences not listed are left as NaN.
    ``threads`` > 1 runs sequences on a thread pool (ctypes releases the GIL).
    """
    q = _c(q, _REAL[q_dtype])
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    out = np.full((B, Hq, D), np.nan, np.float64)
    lib = load()
    seqs = list(range(B)) if seqs is None else [int(s) for s in seqs]

    def run(b):
        return lib.oracle_decode(*cache.args(), _ptr(q), q_dtype, B, Hq, _ptr(bt),
                                 bt.shape[1], _ptr(cl), float(scale), int(window), _ptr(out),
                                 b, b + 1)

    n = _threads(len(seqs), threads)
    if n == 1:
        bad = sum(run(b) for b in seqs)
    else:
        with ThreadPoolExecutor(n) as ex:
            bad = sum(ex.map(run, seqs))
    decode.last_bad = bad
    return out


def prefill(cache: HostCache, q, q_dtype, q_start_loc, block_tables, context_lens, scale,
            *, window=0, seqs=None, threads=None):
    """Chunked-prefill attention in FP64; returns float64 [total_q, Hq, D].  ``window`` > 0:
    each row attends to the last ``window`` positions up to its own."""
    q = _c(q, _REAL[q_dtype])
    qsl = _c(q_start_loc, np.int32)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    Tq, Hq, D = q.shape
    B = cl.shape[0]
    out = np.full((Tq, Hq, D), np.nan, np.float64)
    lib = load()
    seqs = list(range(B)) if seqs is None else [int(s) for s in seqs]

    def run(b):
        return lib.oracle_prefill(*cache.args(), _ptr(q), q_dtype, B, Hq, _ptr(qsl), _ptr(bt),
                                  bt.shape[1], _ptr(cl), float(scale), int(window), _ptr(out),
                                  b, b + 1)

    n = _threads(len(seqs), threads)
    if n == 1:
        bad = sum(run(b) for b in seqs)
    else:
        with ThreadPoolExecutor(n) as ex:
            bad = sum(ex.map(run, seqs))
    prefill.last_bad = bad
    return out


def rope_f64(x, pos, theta):
    """Rotary embedding of one row in double precision (half-split pairs)."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    load().oracle_rope_f64(_ptr(x), _ptr(y), x.shape[0], int(pos), float(theta))
    return y


def rope_f32(x, pos, theta):
    """Rotary embedding of one float32 row in the fixed float operation order used for
    keys that are about to be stored."""
    x = _c(x, np.float32)
    y = np.empty_like(x)
    load().oracle_rope_f32(_ptr(x), _ptr(y), x.shape[0], int(pos), float(theta))
    return y


def decode_step(cache: HostCache, q, q_dtype, k_new, v_new, new_dtype, slot_mapping,
                positions, theta, block_tables, context_lens, scale, *, window=0, seqs=None,
                threads=None):
    """One decode step (rotate, store the new row, attend); mutates ``cache``.

    ``positions`` None: no rotation.  Returns float64 [B, Hq, D]; sequences not listed in
    ``seqs`` are neither stored nor computed (NaN rows).  ``threads`` > 1 runs sequences
    on a thread pool (each stores only its own slot).
    """
    q = _c(q, _REAL[q_dtype])
    k_new = _c(k_new, _REAL[new_dtype])
    v_new = _c(v_new, _REAL[new_dtype])
    sm = _c(slot_mapping, np.int32)
    pos = None if positions is None else _c(positions, np.int32)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    out = np.full((B, Hq, D), np.nan, np.float64)
    lib = load()
    seqs = list(range(B)) if seqs is None else [int(s) for s in seqs]
    def run(b):
        return lib.oracle_decode_step(*cache.args(), _ptr(q), q_dtype, _ptr(k_new), _ptr(v_new),
                                      new_dtype, _ptr(sm), _ptr(pos), float(theta), B, Hq,
                                      _ptr(bt), bt.shape[1], _ptr(cl), float(scale),
                                      int(window), _ptr(out), b, b + 1)

    n = _threads(len(seqs), threads)
    if n == 1:
        bad = sum(run(b) for b in seqs)
    else:
        with ThreadPoolExecutor(n) as ex:
            bad = sum(ex.map(run, seqs))
    decode_step.last_bad = bad
    return out


def cache_from_workload(wl, rows=None, fill=0) -> HostCache:
    """Build the oracle's cache for a workload by appending its source rows."""
    c = HostCache(wl.kv_dtype, wl.num_pages, wl.page_size, wl.num_kv_heads, wl.head_dim, fill)
    sel = slice(None) if rows is None else rows
    append(c, wl.k_src[sel], wl.v_src[sel], wl.new_dtype, wl.slots[sel])
    return c
