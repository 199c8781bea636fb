"""Python binding of libpkv.so: the C ABI of include/pkv.h, same names, argument
marshalling only.  Tensors are torch CUDA tensors (torch supplies device memory and
streams); every computation runs in the library's CUDA kernels.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

F32, BF16, INT8, FP8, INT4 = 0, 1, 2, 3, 4
CODED = (INT8, FP8, INT4)  # stored as codes with one FP32 scale per (token, kv head)
# element containers of the cache tensors (FP8 codes and INT4 code pairs as raw bytes)
# (INT8 bytes hold code + 128, offset binary)
_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, INT8: torch.uint8, FP8: torch.uint8,
                INT4: torch.uint8}
_CODE = {torch.float32: F32, torch.bfloat16: BF16}

DEV_BAD_PAGE, DEV_BAD_LEN, DEV_BAD_SLOT, DEV_BAD_CHUNK, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
STATUS = {0: "PKV_OK", 1: "PKV_ERR_NULL", 2: "PKV_ERR_SHAPE", 3: "PKV_ERR_DTYPE",
          4: "PKV_ERR_PAGE_SIZE", 5: "PKV_ERR_ALIGN", 6: "PKV_ERR_WORKSPACE",
          7: "PKV_ERR_UNSUPPORTED", 8: "PKV_ERR_LAUNCH", 9: "PKV_ERR_DEVICE"}
EXPORTS = ("pkv_append", "pkv_decode_workspace_size", "pkv_decode_attn", "pkv_decode_step",
           "pkv_decode_workspace_size_ex", "pkv_decode_attn_ex", "pkv_decode_step_ex",
           "pkv_prefill_workspace_size", "pkv_prefill_chunk_attn",
           "pkv_prefill_workspace_size_ex", "pkv_prefill_chunk_attn_ex",
           "pkv_decode_attn_noalloc", "pkv_decode_attn_noalloc_ex", "pkv_status_string",
           "pkv_decode_graph_workspace_size", "pkv_decode_graph_create",
           "pkv_decode_graph_launch", "pkv_decode_graph_bucket", "pkv_decode_graph_destroy")
GRAPH_MAX_BUCKETS = 16
NOALLOC_SCRATCH_BYTES = 4 << 20


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class pkv_cache(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("window", ctypes.c_int32)]


class pkv_decode_opts(ctypes.Structure):
    _fields_ = [("split_pages", ctypes.c_int32)]


class pkv_prefill_opts(ctypes.Structure):
    _fields_ = [("key_split", ctypes.c_int32)]


class pkv_graph_layer(ctypes.Structure):
    _fields_ = [("cache", pkv_cache), ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class pkv_decode_graph_desc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("layers", ctypes.POINTER(pkv_graph_layer)),
                ("num_q_heads", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
                ("new_dtype", ctypes.c_int32), ("fused", ctypes.c_int32),
                ("block_tables", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int32),
                ("context_lens", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
                ("positions", ctypes.c_void_p), ("rope_theta", ctypes.c_double),
                ("scale", ctypes.c_float), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p),
                ("num_buckets", ctypes.c_int32), ("buckets", ctypes.POINTER(ctypes.c_int32))]


_lib = None


def load(path: str = LIB_PATH):
    """Load libpkv.so (build it with __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = bind(path)
    return _lib


def bind(path: str):
    """A handle on the library at ``path`` with every entry point's argument types (a
    variant build, e.g. a test build, is used beside the product library this way)."""
    if not os.path.exists(path):
        raise RuntimeError(f"libpkv.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    C = ctypes.POINTER(pkv_cache)
    lib.pkv_append.argtypes = [C, P, P, I32, P, I32, P, P]
    O = ctypes.POINTER(pkv_decode_opts)
    lib.pkv_decode_workspace_size.argtypes = [C, I32, I32, I32, ctypes.POINTER(SZ)]
    lib.pkv_decode_workspace_size_ex.argtypes = [C, I32, I32, I32, O, ctypes.POINTER(SZ)]
    lib.pkv_decode_attn.argtypes = [C, P, I32, I32, I32, P, I32, P, F, P, P, SZ, P, P]
    lib.pkv_decode_attn_ex.argtypes = [C, P, I32, I32, I32, P, I32, P, F, P, P, SZ, O, P, P]
    lib.pkv_decode_step.argtypes = [C, P, I32, P, P, I32, P, P, ctypes.c_double, I32, I32, P,
                                    I32, P, F, P, P, SZ, P, P]
    lib.pkv_decode_step_ex.argtypes = [C, P, I32, P, P, I32, P, P, ctypes.c_double, I32, I32,
                                       P, I32, P, F, P, P, SZ, O, P, P]
    lib.pkv_prefill_workspace_size.argtypes = [C, I32, I32, I32, I32, ctypes.POINTER(SZ)]
    lib.pkv_prefill_chunk_attn.argtypes = [C, P, I32, I32, I32, P, I32, P, I32, P, F, P, P, SZ,
                                           P, P]
    PO = ctypes.POINTER(pkv_prefill_opts)
    lib.pkv_prefill_workspace_size_ex.argtypes = [C, I32, I32, I32, I32, PO, ctypes.POINTER(SZ)]
    lib.pkv_prefill_chunk_attn_ex.argtypes = [C, P, I32, I32, I32, P, I32, P, I32, P, F, P, P,
                                              SZ, PO, P, P]
    for fn in ("pkv_append", "pkv_decode_workspace_size", "pkv_decode_attn", "pkv_decode_step",
               "pkv_decode_workspace_size_ex", "pkv_decode_attn_ex", "pkv_decode_step_ex",
               "pkv_prefill_workspace_size", "pkv_prefill_chunk_attn",
               "pkv_prefill_workspace_size_ex", "pkv_prefill_chunk_attn_ex"):
        getattr(lib, fn).restype = ctypes.c_int
    lib.pkv_decode_attn_noalloc.argtypes = [C, P, I32, I32, I32, P, I32, P, F, P, P, P]
    lib.pkv_decode_attn_noalloc.restype = ctypes.c_int
    lib.pkv_decode_attn_noalloc_ex.argtypes = [C, P, I32, I32, I32, P, I32, P, F, P, O, P, P]
    lib.pkv_decode_attn_noalloc_ex.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    GD = ctypes.POINTER(pkv_decode_graph_desc)
    lib.pkv_decode_graph_workspace_size.argtypes = [GD, ctypes.POINTER(SZ)]
    lib.pkv_decode_graph_create.argtypes = [GD, ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_decode_graph_launch.argtypes = [P, I32, P]
    lib.pkv_decode_graph_bucket.argtypes = [P, I32]
    lib.pkv_decode_graph_destroy.argtypes = [P]
    lib.pkv_decode_graph_destroy.restype = None
    for fn in ("pkv_decode_graph_workspace_size", "pkv_decode_graph_create",
               "pkv_decode_graph_launch", "pkv_decode_graph_bucket"):
        getattr(lib, fn).restype = ctypes.c_int
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(code: int, what: str):
    if code != 0:
        raise PkvError(code, what)


class BoundCall:
    """One library call with its arguments marshalled once: the cache struct, device
    pointers, sizes, options and stream.  Calling it issues the same C call again, with no
    Python work beyond the ctypes call itself (about a microsecond against ~10 for the
    full wrapper), for loops that repeat a launch on fixed buffers.  The caller keeps the
    tensors alive and their contents current; a non-zero status raises PkvError."""

    __slots__ = ("_fn", "_args", "_what")

    def __init__(self, fn, args, what: str):
        self._fn, self._args, self._what = fn, tuple(args), what

    def __call__(self) -> None:
        code = self._fn(*self._args)
        if code != 0:
            raise PkvError(code, self._what)


def _call(fn, args, what: str, bound: bool):
    """Issue the call now, or (bound=True) return it as a BoundCall without issuing it."""
    if bound:
        return BoundCall(fn, args, what)
    _check(fn(*args), what)
    return None


class KVCache:
    """Device tensors of one paged cache in the library's layout.

    k: [num_pages, Hkv, 16, D]; v: [num_pages, Hkv, D, 16] (page blocks transposed);
    k_scale, v_scale: float32 [num_pages, Hkv, 16] for INT8, FP8 and INT4 caches.  For
    BF16 caches the elements inside each (page, kv head) block are in tensor-core tile
    order, FP8 codes are bytes, and INT4 blocks hold two codes per byte (k: [.., 16, D/2],
    v: [.., D/2, 16] bytes); see include/pkv.h.  The tensor shapes are containers of the
    right size.
    """

    def __init__(self, k, v, k_scale=None, v_scale=None, window=0, kv_dtype=None):
        self.k, self.v, self.k_scale, self.v_scale = k, v, k_scale, v_scale
        self.kv_dtype = _CODE[k.dtype] if kv_dtype is None else int(kv_dtype)
        self.num_pages, self.num_kv_heads, self.page_size, self.head_dim = k.shape
        if self.kv_dtype == INT4:
            self.head_dim *= 2
        self.window = int(window)  # sliding window in tokens (0: none), read by every call

    @classmethod
    def allocate(cls, num_pages, num_kv_heads, head_dim, kv_dtype, device="cuda",
                 page_size=16):
        dt = _TORCH_DTYPE[kv_dtype]
        if kv_dtype == INT4:
            k = torch.zeros(num_pages, num_kv_heads, page_size, head_dim // 2, dtype=dt, device=device)
            v = torch.zeros(num_pages, num_kv_heads, head_dim // 2, page_size, dtype=dt, device=device)
        else:
            k = torch.zeros(num_pages, num_kv_heads, page_size, head_dim, dtype=dt, device=device)
            v = torch.zeros(num_pages, num_kv_heads, head_dim, page_size, dtype=dt, device=device)
        ks = vs = None
        if kv_dtype in CODED:
            ks = torch.zeros(num_pages, num_kv_heads, page_size, dtype=torch.float32, device=device)
            vs = torch.zeros_like(ks)
        return cls(k, v, ks, vs, kv_dtype=kv_dtype)

    def clone(self) -> "KVCache":
        """A copy in fresh device memory (same format and window)."""
        return KVCache(self.k.clone(), self.v.clone(),
                       None if self.k_scale is None else self.k_scale.clone(),
                       None if self.v_scale is None else self.v_scale.clone(),
                       window=self.window, kv_dtype=self.kv_dtype)

    def struct(self) -> pkv_cache:
        return pkv_cache(self.k.data_ptr(), self.v.data_ptr(),
                         None if self.k_scale is None else self.k_scale.data_ptr(),
                         None if self.v_scale is None else self.v_scale.data_ptr(),
                         self.num_pages, self.page_size, self.num_kv_heads, self.head_dim,
                         self.kv_dtype, self.window)


def pkv_status_string(code: int) -> str:
    return load().pkv_status_string(code).decode()


def _opts(split_pages: int):
    """The options argument of the _ex calls (None: every option at its default)."""
    return None if not split_pages else ctypes.byref(pkv_decode_opts(int(split_pages)))


def pkv_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
               slot_mapping: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
               stream=None, bound: bool = False) -> Optional[BoundCall]:
    c = cache.struct()
    return _call(load().pkv_append,
                 (ctypes.byref(c), _ptr(k_new), _ptr(v_new), _CODE[k_new.dtype],
                  _ptr(slot_mapping), int(slot_mapping.shape[0]), _ptr(dev_status),
                  _stream(stream)), "pkv_append", bound)


def pkv_decode_workspace_size(cache: KVCache, num_seqs: int, num_q_heads: int,
                              max_blocks_per_seq: int, split_pages: int = 0) -> int:
    """Scratch bytes of the decode calls for this shape; ``split_pages`` as in
    pkv_decode_opts (0: automatic)."""
    c = cache.struct()
    n = ctypes.c_size_t(0)
    _check(load().pkv_decode_workspace_size_ex(ctypes.byref(c), num_seqs, num_q_heads,
                                               max_blocks_per_seq, _opts(split_pages),
                                               ctypes.byref(n)),
           "pkv_decode_workspace_size")
    return int(n.value)


def pkv_decode_attn(cache: KVCache, q: torch.Tensor, block_tables: torch.Tensor,
                    context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                    workspace: Optional[torch.Tensor] = None,
                    dev_status: Optional[torch.Tensor] = None, stream=None,
                    split_pages: int = 0, bound: bool = False) -> Optional[BoundCall]:
    c = cache.struct()
    B, Hq, _ = q.shape
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _call(load().pkv_decode_attn_ex,
                 (ctypes.byref(c), _ptr(q), _CODE[q.dtype], B, Hq, _ptr(block_tables),
                  int(block_tables.shape[1]), _ptr(context_lens), float(scale), _ptr(out),
                  _ptr(workspace), wb, _opts(split_pages), _ptr(dev_status), _stream(stream)),
                 "pkv_decode_attn", bound)


def pkv_decode_step(cache: KVCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    slot_mapping: torch.Tensor, positions: Optional[torch.Tensor],
                    rope_theta: float, block_tables: torch.Tensor, context_lens: torch.Tensor,
                    scale: float, out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                    dev_status: Optional[torch.Tensor] = None, stream=None,
                    split_pages: int = 0, bound: bool = False) -> Optional[BoundCall]:
    """One fused decode step (rotate, append the new row, attend); see include/pkv.h."""
    c = cache.struct()
    B, Hq, _ = q.shape
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _call(load().pkv_decode_step_ex,
                 (ctypes.byref(c), _ptr(q), _CODE[q.dtype], _ptr(k_new), _ptr(v_new),
                  _CODE[k_new.dtype], _ptr(slot_mapping), _ptr(positions), float(rope_theta),
                  B, Hq, _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
                  float(scale), _ptr(out), _ptr(workspace), wb, _opts(split_pages),
                  _ptr(dev_status), _stream(stream)), "pkv_decode_step", bound)


class GraphLayer:
    """One layer of a decode-graph step: its cache, query rows, new K/V rows (or None: no
    append) and output, all sized for the largest bucket."""

    def __init__(self, cache: KVCache, q: torch.Tensor, out: torch.Tensor,
                 k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None):
        self.cache, self.q, self.out, self.k_new, self.v_new = cache, q, out, k_new, v_new


class DecodeGraph:
    """pkv_decode_graph: one captured CUDA graph per batch-size bucket (see include/pkv.h).

    The tensors are captured by address and must stay alive (and in place) for the
    executor's lifetime; rows past a launch's num_seqs up to its bucket must be inert
    (context_lens 0, slot_mapping -1).  The workspace is allocated here, zero-filled."""

    def __init__(self, layers, block_tables: torch.Tensor, context_lens: torch.Tensor,
                 scale: float, buckets, slot_mapping: Optional[torch.Tensor] = None,
                 fused: bool = False, positions: Optional[torch.Tensor] = None,
                 rope_theta: float = 10000.0, dev_status: Optional[torch.Tensor] = None):
        lib = load()
        self.layers = list(layers)
        self._keep = (block_tables, context_lens, slot_mapping, positions, dev_status)
        arr = (pkv_graph_layer * len(self.layers))()
        for i, L in enumerate(self.layers):
            arr[i] = pkv_graph_layer(L.cache.struct(), _ptr(L.q), _ptr(L.k_new), _ptr(L.v_new),
                                     _ptr(L.out))
        self._arr = arr
        self._buckets = (ctypes.c_int32 * len(buckets))(*[int(b) for b in buckets])
        q0 = self.layers[0].q
        k0 = next((L.k_new for L in self.layers if L.k_new is not None), None)
        d = pkv_decode_graph_desc()
        d.num_layers = len(self.layers)
        d.layers = ctypes.cast(arr, ctypes.POINTER(pkv_graph_layer))
        d.num_q_heads = int(q0.shape[1])
        d.q_dtype = _CODE[q0.dtype]
        d.new_dtype = _CODE[k0.dtype] if k0 is not None else F32
        d.fused = 1 if fused else 0
        d.block_tables = _ptr(block_tables)
        d.max_blocks_per_seq = int(block_tables.shape[1])
        d.context_lens = _ptr(context_lens)
        d.slot_mapping = _ptr(slot_mapping)
        d.positions = _ptr(positions)
        d.rope_theta = float(rope_theta)
        d.scale = float(scale)
        d.dev_status = _ptr(dev_status)
        d.num_buckets = len(buckets)
        d.buckets = ctypes.cast(self._buckets, ctypes.POINTER(ctypes.c_int32))
        n = ctypes.c_size_t(0)
        _check(lib.pkv_decode_graph_workspace_size(ctypes.byref(d), ctypes.byref(n)),
               "pkv_decode_graph_workspace_size")
        self.workspace = workspace_for(int(n.value), q0.device)
        d.workspace = _ptr(self.workspace)
        d.workspace_bytes = int(n.value)
        self._desc = d
        h = ctypes.c_void_p(None)
        _check(lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)),
               "pkv_decode_graph_create")
        self._h = h

    def bucket(self, num_seqs: int) -> int:
        return int(load().pkv_decode_graph_bucket(self._h, int(num_seqs)))

    def launch(self, num_seqs: int, stream=None) -> None:
        _check(load().pkv_decode_graph_launch(self._h, int(num_seqs), _stream(stream)),
               "pkv_decode_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            load().pkv_decode_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pkv_decode_attn_noalloc(cache: KVCache, q: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                            dev_status: Optional[torch.Tensor] = None, stream=None,
                            split_pages: int = 0) -> None:
    """pkv_decode_attn with its split scratch in the library's fixed device array (for
    callers that cannot allocate); see include/pkv.h for the size limit and sharing."""
    c = cache.struct()
    B, Hq, _ = q.shape
    _check(load().pkv_decode_attn_noalloc_ex(ctypes.byref(c), _ptr(q), _CODE[q.dtype], B, Hq,
                                             _ptr(block_tables), int(block_tables.shape[1]),
                                             _ptr(context_lens), float(scale), _ptr(out),
                                             _opts(split_pages), _ptr(dev_status),
                                             _stream(stream)),
           "pkv_decode_attn_noalloc")


def _prefill_opts(key_split: int):
    """The options argument of the prefill _ex calls (None: every option at its default)."""
    return None if not key_split else ctypes.byref(pkv_prefill_opts(int(key_split)))


def pkv_prefill_workspace_size(cache: KVCache, num_seqs: int, num_q_heads: int,
                               max_q_len: int, max_blocks_per_seq: int,
                               key_split: int = 0) -> int:
    """Scratch bytes of pkv_prefill_chunk_attn; key_split (0: automatic, 1..3) is the
    pkv_prefill_opts option."""
    c = cache.struct()
    n = ctypes.c_size_t(0)
    _check(load().pkv_prefill_workspace_size_ex(ctypes.byref(c), num_seqs, num_q_heads,
                                                max_q_len, max_blocks_per_seq,
                                                _prefill_opts(key_split), ctypes.byref(n)),
           "pkv_prefill_workspace_size")
    return int(n.value)


def pkv_prefill_chunk_attn(cache: KVCache, q: torch.Tensor, q_start_loc: torch.Tensor,
                           max_q_len: int, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                           workspace: Optional[torch.Tensor] = None,
                           dev_status: Optional[torch.Tensor] = None, stream=None,
                           key_split: int = 0, bound: bool = False) -> Optional[BoundCall]:
    c = cache.struct()
    B = int(context_lens.shape[0])
    Hq = int(q.shape[1])
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _call(load().pkv_prefill_chunk_attn_ex,
                 (ctypes.byref(c), _ptr(q), _CODE[q.dtype], B, Hq, _ptr(q_start_loc),
                  int(max_q_len), _ptr(block_tables), int(block_tables.shape[1]),
                  _ptr(context_lens), float(scale), _ptr(out), _ptr(workspace), wb,
                  _prefill_opts(key_split), _ptr(dev_status), _stream(stream)),
                 "pkv_prefill_chunk_attn", bound)


def workspace_for(nbytes: int, device="cuda") -> Optional[torch.Tensor]:
    """A zero-filled workspace tensor of at least nbytes (16-byte aligned), or None."""
    if nbytes == 0:
        return None
    return torch.zeros((nbytes + 15) // 16 * 4, dtype=torch.int32, device=device)
