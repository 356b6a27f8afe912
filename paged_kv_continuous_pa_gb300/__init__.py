"""Python binding of libpa_gb300 (include/pa.h): argument marshalling only.

Every step of append and attention runs in the library's CUDA kernels; this
module passes tensor pointers, sizes and the current CUDA stream through
ctypes.  PyTorch supplies device memory and streams.  There is no fallback:
if the shared library is missing or a CUDA device is absent the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional, Sequence, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libpa_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pa.h")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_RANGE, PA_ERR_TIMEOUT, PA_ERR_CUDA, PA_ERR_NO_PAGES = range(7)
PA_ADMIT_OK, PA_ADMIT_NO_PAGES, PA_ADMIT_TOO_LONG, PA_ADMIT_SEQ_IN_USE, PA_ADMIT_BAD_ARG = range(5)
PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_ORDER_AUTO, PA_ORDER_CALL, PA_ORDER_LONGEST_FIRST = 0, 1, 2

_lib = None
_lock = threading.Lock()


class PaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{status_string(status) if _lib else status}: {detail}")


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class Chunk(ctypes.Structure):
    _fields_ = [("row_begin", ctypes.c_int32), ("n_rows", ctypes.c_int32)]


class AdmitInfo(ctypes.Structure):
    _fields_ = [("reason", ctypes.c_int32), ("pages_needed", ctypes.c_int32), ("pages_free", ctypes.c_int32),
                ("pages_shared", ctypes.c_int32), ("tokens", ctypes.c_int32), ("max_tokens", ctypes.c_int32)]


def header_functions():
    """Names of the functions include/pa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Load the shared library and declare the C signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libpa_gb300.so not built at {path}; run paged_kv_continuous_pa_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        st = ctypes.c_int
        L.pa_pool_bytes.argtypes = [ctypes.POINTER(PoolDesc)]
        L.pa_pool_bytes.restype = sz
        L.pa_pool_create.argtypes = [ctypes.POINTER(PoolDesc), vp, vp, ctypes.POINTER(vp)]
        L.pa_pool_create.restype = st
        L.pa_pool_destroy.argtypes = [vp]
        L.pa_pool_destroy.restype = None
        L.pa_pool_set_head_scales.argtypes = [vp, vp, vp]
        L.pa_pool_set_head_scales.restype = st
        L.pa_append_kv.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, i32, i32, vp, vp]
        L.pa_append_kv.restype = st
        L.pa_attention_workspace_bytes.argtypes = [vp, i32, i32, i32, ctypes.POINTER(Chunk), i32]
        L.pa_attention_workspace_bytes.restype = sz
        L.pa_attention.argtypes = [vp, i32, vp, i32, i32, vp, vp, vp, i32, i32, ctypes.POINTER(Chunk), i32, f32, vp,
                                   vp, sz, vp, vp]
        L.pa_attention.restype = st
        L.pa_attention_noalloc.argtypes = [vp, i32, vp, i32, i32, vp, vp, vp, i32, i32, ctypes.POINTER(Chunk), i32,
                                           f32, vp, vp, vp]
        L.pa_attention_noalloc.restype = st
        L.pa_step.argtypes = [vp, i32, vp, i32, i32, vp, vp, i32, vp, vp, vp, i32, i32, ctypes.POINTER(Chunk), i32,
                              f32, vp, vp, sz, vp, vp]
        L.pa_step.restype = st
        L.pa_pages_needed.argtypes = [i32, i32, i32]
        L.pa_pages_needed.restype = i32
        L.pa_pages_create.argtypes = [i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.pa_pages_create.restype = st
        L.pa_pages_destroy.argtypes = [vp]
        L.pa_pages_destroy.restype = None
        L.pa_pages_admit.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.POINTER(AdmitInfo)]
        L.pa_pages_admit.restype = st
        L.pa_pages_release.argtypes = [vp, i32, vp]
        L.pa_pages_release.restype = st
        L.pa_pages_free_count.argtypes = [vp]
        L.pa_pages_free_count.restype = i32
        L.pa_pages_refcount.argtypes = [vp, i32]
        L.pa_pages_refcount.restype = i32
        L.pa_set_split_tokens.argtypes = [i32]
        L.pa_set_split_tokens.restype = st
        L.pa_get_split_tokens.argtypes = []
        L.pa_get_split_tokens.restype = i32
        L.pa_set_row_groups.argtypes = [i32]
        L.pa_set_row_groups.restype = st
        L.pa_get_row_groups.argtypes = []
        L.pa_get_row_groups.restype = i32
        L.pa_set_unit_order.argtypes = [i32]
        L.pa_set_unit_order.restype = st
        L.pa_get_unit_order.argtypes = []
        L.pa_get_unit_order.restype = i32
        L.pa_set_wait_limit.argtypes = [ctypes.c_uint32]
        L.pa_set_wait_limit.restype = None
        L.pa_debug_stall_waits.argtypes = [i32]
        L.pa_debug_stall_waits.restype = None
        L.pa_status_string.argtypes = [st]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_last_error.argtypes = []
        L.pa_last_error.restype = ctypes.c_char_p
        L.pa_kernel_launches.argtypes = []
        L.pa_kernel_launches.restype = ctypes.c_uint64
        L.pa_version.argtypes = []
        L.pa_version.restype = ctypes.c_char_p
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def last_error() -> str:
    return load().pa_last_error().decode()


def _check(status: int):
    if status != PA_OK:
        raise PaError(status, last_error())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return PA_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _check_index(t, name: str, n: Optional[int] = None, dims: int = 1):
    """The int32 index arrays the kernels read: dtype and shape, before any pointer is taken."""
    import torch
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32, got {t.dtype}")
    if t.dim() != dims or (n is not None and int(t.shape[0]) != n):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {dims}-D" + (f" with {n} rows" if n is not None else ""))


def _check_rows(pool: "Pool", q, seq_ids, positions, block_tables, out, status):
    """q / out [n, Hq, D] with the pool's D; seq_ids / positions int32 [n]; block_tables int32 [num_seqs, max_blocks]."""
    _check_index(seq_ids, "seq_ids")
    n = int(seq_ids.shape[0])
    _check_index(positions, "positions", n)
    _check_index(block_tables, "block_tables", dims=2)
    if status is not None:
        _check_index(status, "status")
    if q.dim() != 3 or int(q.shape[0]) != n or int(q.shape[2]) != pool.head_dim:
        raise ValueError(f"q has shape {tuple(q.shape)}; expected [{n}, Hq, {pool.head_dim}]")
    if out.dtype != q.dtype or tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must match q's shape and dtype")
    return n


def _check_kv_rows(pool: "Pool", k_new, v_new, n: int):
    """k_new / v_new [n, Hkv, D] with the pool's Hkv and D, one dtype."""
    want = (n, pool.num_kv_heads, pool.head_dim)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if tuple(t.shape) != want:
            raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {list(want)}")
    if k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must share a dtype")


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pool_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int, kv_dtype: int,
               k_scale: float = 1.0, v_scale: float = 1.0) -> int:
    d = PoolDesc(num_pages, page_size, num_kv_heads, head_dim, kv_dtype, k_scale, v_scale)
    return int(load().pa_pool_bytes(ctypes.byref(d)))


class Pool:
    """A paged K/V pool over two caller-owned device tensors [num_pages, Hkv, P, D]."""

    def __init__(self, k_pool, v_pool, k_scale=1.0, v_scale=1.0):
        """k_scale / v_scale: fp8 scales, one float (per tensor) or one per kv head."""
        import numpy as np
        if k_pool.shape != v_pool.shape or k_pool.dim() != 4 or k_pool.dtype != v_pool.dtype:
            raise ValueError("k_pool and v_pool must be matching [num_pages, Hkv, P, D] tensors")
        self.k_pool, self.v_pool = k_pool, v_pool
        n, h, p, d = k_pool.shape
        self.num_pages, self.num_kv_heads, self.page_size, self.head_dim = int(n), int(h), int(p), int(d)
        self.kv_dtype = _dtype_code(k_pool)
        per_head = np.ndim(k_scale) > 0 or np.ndim(v_scale) > 0
        self.k_scale = np.asarray(k_scale, np.float32) if per_head else float(k_scale)
        self.v_scale = np.asarray(v_scale, np.float32) if per_head else float(v_scale)
        self.desc = PoolDesc(self.num_pages, self.page_size, self.num_kv_heads, self.head_dim, self.kv_dtype,
                             1.0 if per_head else self.k_scale, 1.0 if per_head else self.v_scale)
        handle = ctypes.c_void_p()
        _check(load().pa_pool_create(ctypes.byref(self.desc), _ptr(k_pool), _ptr(v_pool), ctypes.byref(handle)))
        self._h = handle
        if per_head:
            ks = np.ascontiguousarray(np.broadcast_to(self.k_scale, (self.num_kv_heads,)), np.float32)
            vs = np.ascontiguousarray(np.broadcast_to(self.v_scale, (self.num_kv_heads,)), np.float32)
            _check(load().pa_pool_set_head_scales(self._h, ks.ctypes.data_as(ctypes.c_void_p),
                                                  vs.ctypes.data_as(ctypes.c_void_p)))

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().pa_pool_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def pages_needed(page_size: int, prompt_tokens: int, max_new_tokens: int) -> int:
    """Pages a sequence of prompt + answer tokens needs (no allocation)."""
    return int(load().pa_pages_needed(int(page_size), int(prompt_tokens), int(max_new_tokens)))


class Pages:
    """Host page allocator with admission over one pool's page ids; owns the host
    block-table array int32 [num_seqs, max_blocks] (numpy) whose rows it fills."""

    def __init__(self, num_pages: int, page_size: int, num_seqs: int, max_blocks: int):
        import numpy as np
        h = ctypes.c_void_p()
        _check(load().pa_pages_create(int(num_pages), int(page_size), int(num_seqs), int(max_blocks), ctypes.byref(h)))
        self.handle = h
        self.page_size = int(page_size)
        self.block_tables = np.full((int(num_seqs), int(max_blocks)), -1, dtype=np.int32)

    def admit(self, seq: int, prompt_tokens: int, max_new_tokens: int, prefix_parent: int = -1,
              prefix_tokens: int = 0):
        """(status, AdmitInfo); the slot's row of block_tables is filled on PA_OK."""
        info = AdmitInfo()
        st = load().pa_pages_admit(self.handle, int(seq), int(prompt_tokens), int(max_new_tokens), int(prefix_parent),
                                   int(prefix_tokens), self.block_tables.ctypes.data_as(ctypes.c_void_p),
                                   ctypes.byref(info))
        return int(st), info

    def release(self, seq: int):
        _check(load().pa_pages_release(self.handle, int(seq), self.block_tables.ctypes.data_as(ctypes.c_void_p)))

    def free_count(self) -> int:
        return int(load().pa_pages_free_count(self.handle))

    def refcount(self, page: int) -> int:
        return int(load().pa_pages_refcount(self.handle, int(page)))

    def __del__(self):
        try:
            if _lib is not None and getattr(self, "handle", None):
                _lib.pa_pages_destroy(self.handle)
        except Exception:
            pass


def append_kv(pool: Pool, k_new, v_new, seq_ids, positions, block_tables, status=None, stream=None):
    """Scatter rows' new K/V ([n, Hkv, D], f32 or bf16) into their page slots (one launch)."""
    _check_index(seq_ids, "seq_ids")
    n = int(seq_ids.shape[0])
    _check_index(positions, "positions", n)
    _check_index(block_tables, "block_tables", dims=2)
    if status is not None:
        _check_index(status, "status")
    _check_kv_rows(pool, k_new, v_new, n)
    num_seqs, max_blocks = (int(x) for x in block_tables.shape)
    _check(load().pa_append_kv(pool.handle, n, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(seq_ids),
                               _ptr(positions), _ptr(block_tables), num_seqs, max_blocks, _ptr(status),
                               _stream(stream)))


def workspace_bytes(pool: Pool, n_rows: int, num_q_heads: int, max_blocks: int,
                    chunks: Sequence[Tuple[int, int]] = ()) -> int:
    arr = (Chunk * max(1, len(chunks)))(*[Chunk(int(b), int(c)) for b, c in chunks])
    return int(load().pa_attention_workspace_bytes(pool.handle, int(n_rows), int(num_q_heads), int(max_blocks),
                                                   arr if chunks else None, len(chunks)))


def attention(pool: Pool, q, seq_ids, positions, block_tables, out,
              chunks: Sequence[Tuple[int, int]] = (), softmax_scale: float = 0.0, workspace=None, status=None,
              stream=None):
    """Paged attention of every row (q [n, Hq, D] f32|bf16) into out (same shape and dtype)."""
    n = _check_rows(pool, q, seq_ids, positions, block_tables, out, status)
    num_q_heads = int(q.shape[1])
    num_seqs, max_blocks = (int(x) for x in block_tables.shape)
    arr = (Chunk * max(1, len(chunks)))(*[Chunk(int(b), int(c)) for b, c in chunks])
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_attention(pool.handle, n, _ptr(q), _dtype_code(q), num_q_heads, _ptr(seq_ids), _ptr(positions),
                               _ptr(block_tables), num_seqs, max_blocks, arr if chunks else None, len(chunks),
                               float(softmax_scale), _ptr(out), ws_ptr, ws_len, _ptr(status), _stream(stream)))


def step(pool: Pool, q, k_new, v_new, seq_ids, positions, block_tables, out,
         chunks: Sequence[Tuple[int, int]] = (), softmax_scale: float = 0.0, workspace=None, status=None, stream=None):
    """append_kv() then attention() of the same rows as one call: the attention
    kernel starts while the append runs (bit-identical to the two calls)."""
    n = _check_rows(pool, q, seq_ids, positions, block_tables, out, status)
    _check_kv_rows(pool, k_new, v_new, n)
    num_q_heads = int(q.shape[1])
    num_seqs, max_blocks = (int(x) for x in block_tables.shape)
    arr = (Chunk * max(1, len(chunks)))(*[Chunk(int(b), int(c)) for b, c in chunks])
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_step(pool.handle, n, _ptr(q), _dtype_code(q), num_q_heads, _ptr(k_new), _ptr(v_new),
                          _dtype_code(k_new), _ptr(seq_ids), _ptr(positions), _ptr(block_tables), num_seqs, max_blocks,
                          arr if chunks else None, len(chunks), float(softmax_scale), _ptr(out), ws_ptr, ws_len,
                          _ptr(status), _stream(stream)))


def attention_noalloc(pool: Pool, q, seq_ids, positions, block_tables, out,
                      chunks: Sequence[Tuple[int, int]] = (), softmax_scale: float = 0.0, status=None, stream=None):
    """attention() for callers that cannot allocate: split-KV scratch comes from
    a fixed 32 MiB array inside the library instead of a workspace tensor."""
    n = _check_rows(pool, q, seq_ids, positions, block_tables, out, status)
    num_q_heads = int(q.shape[1])
    num_seqs, max_blocks = (int(x) for x in block_tables.shape)
    arr = (Chunk * max(1, len(chunks)))(*[Chunk(int(b), int(c)) for b, c in chunks])
    _check(load().pa_attention_noalloc(pool.handle, n, _ptr(q), _dtype_code(q), num_q_heads, _ptr(seq_ids),
                                       _ptr(positions), _ptr(block_tables), num_seqs, max_blocks,
                                       arr if chunks else None, len(chunks), float(softmax_scale), _ptr(out),
                                       _ptr(status), _stream(stream)))


def set_split_tokens(tokens: int):
    _check(load().pa_set_split_tokens(int(tokens)))


def get_split_tokens() -> int:
    return int(load().pa_get_split_tokens())


def set_row_groups(rows: int):
    _check(load().pa_set_row_groups(int(rows)))


def get_row_groups() -> int:
    return int(load().pa_get_row_groups())


def set_unit_order(mode: int):
    _check(load().pa_set_unit_order(int(mode)))


def get_unit_order() -> int:
    return int(load().pa_get_unit_order())


def set_wait_limit(microseconds: int):
    load().pa_set_wait_limit(int(microseconds))


def kernel_launches() -> int:
    return int(load().pa_kernel_launches())


def debug_stall_waits(enable: bool):
    load().pa_debug_stall_waits(1 if enable else 0)


def version() -> str:
    return load().pa_version().decode()
