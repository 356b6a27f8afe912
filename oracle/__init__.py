"""The CPU oracle: test infrastructure, not product code.

A plain FP64 C implementation (``oracle.c``) of paged K/V append and paged
attention, loaded through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU legs of ``bench.py`` may import this package; the CUDA library in
``paged_kv_continuous_pa_gb300`` shares no code with it and never calls it.

Arrays are numpy: f32 data as ``float32``, bf16 data as ``uint16`` bit
patterns, fp8 e4m3 data as ``uint8`` codes.  Pools are flat byte-compatible
arrays laid out ``[num_pages][Hkv][P][D]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

F32, BF16, E4M3 = 0, 1, 2
_NP_OF = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (no fast-math, no FP contraction)."""
    src = os.path.join(HERE, "oracle.c")
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(src):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load(path: str):
    """Load an oracle shared library at path and declare its C signatures."""
    L = ctypes.CDLL(path)
    i32, f32, f64, vp = ctypes.c_int32, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
    L.oracle_bf16_from_f32.argtypes = [f32]
    L.oracle_bf16_from_f32.restype = ctypes.c_uint16
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f64.restype = f64
    L.oracle_e4m3_from_f32.argtypes = [f32]
    L.oracle_e4m3_from_f32.restype = ctypes.c_uint8
    L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f64.restype = f64
    L.oracle_e4m3_from_f32_array.argtypes = [vp, vp, ctypes.c_int64]
    L.oracle_e4m3_from_f32_array.restype = None
    L.oracle_append.argtypes = [i32, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                i32, f32, f32, vp, vp]
    L.oracle_append.restype = ctypes.c_int
    L.oracle_attention.argtypes = [i32, vp, i32, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                   i32, i32, f32, f32, vp, vp, f64, vp, i32]
    L.oracle_attention.restype = ctypes.c_int
    L.oracle_append_h.argtypes = [i32, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    L.oracle_append_h.restype = ctypes.c_int
    L.oracle_attention_h.argtypes = [i32, vp, i32, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                     vp, f64, vp, i32]
    L.oracle_attention_h.restype = ctypes.c_int
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load(LIB_PATH)
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_from_f32(x: float) -> int:
    return int(lib().oracle_bf16_from_f32(float(x)))


def bf16_to_f64(h: int) -> float:
    return float(lib().oracle_bf16_to_f64(int(h)))


def e4m3_from_f32(x: float) -> int:
    return int(lib().oracle_e4m3_from_f32(float(x)))


def e4m3_to_f64(code: int) -> float:
    return float(lib().oracle_e4m3_to_f64(int(code)))


def e4m3_from_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_from_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def decode_pool(pool: np.ndarray, kv_dtype: int, scale: float = 1.0) -> np.ndarray:
    """Stored pool elements as float64 (fp8 codes times their scale), element by element."""
    flat = np.ascontiguousarray(pool).reshape(-1)
    if kv_dtype == F32:
        return flat.view(np.float32).astype(np.float64).reshape(pool.shape)
    if kv_dtype == BF16:
        return (flat.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(pool.shape)
    table = np.array([lib().oracle_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
    return (table[flat.view(np.uint8)] * np.float64(scale)).reshape(pool.shape)


def _head_scales(scale, num_kv_heads: int) -> np.ndarray:
    """A scale per kv head as float32 (a scalar repeated)."""
    s = np.ascontiguousarray(np.broadcast_to(np.asarray(scale, dtype=np.float32), (num_kv_heads,)))
    return s.copy()


def append(k_new, v_new, in_dtype, seq_ids, positions, block_tables, num_pages, page_size,
           num_kv_heads, head_dim, kv_dtype, k_scale, v_scale, k_pool, v_pool) -> int:
    """Scatter rows into the pools in place (row order).  Returns the C status (0 = ok)."""
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    seq_ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    assert k_new.dtype == _NP_OF[in_dtype] and v_new.dtype == _NP_OF[in_dtype]
    assert k_pool.dtype == _NP_OF[kv_dtype] and v_pool.dtype == _NP_OF[kv_dtype]
    num_seqs, max_blocks = block_tables.shape
    if np.ndim(k_scale) or np.ndim(v_scale):  # one scale per kv head
        ks, vs = _head_scales(k_scale, num_kv_heads), _head_scales(v_scale, num_kv_heads)
        return int(lib().oracle_append_h(int(seq_ids.shape[0]), _ptr(k_new), _ptr(v_new), in_dtype,
                                         _ptr(seq_ids), _ptr(positions), _ptr(block_tables), num_seqs,
                                         max_blocks, num_pages, page_size, num_kv_heads, head_dim,
                                         kv_dtype, _ptr(ks), _ptr(vs), _ptr(k_pool), _ptr(v_pool)))
    return int(lib().oracle_append(int(seq_ids.shape[0]), _ptr(k_new), _ptr(v_new), in_dtype,
                                   _ptr(seq_ids), _ptr(positions), _ptr(block_tables), num_seqs,
                                   max_blocks, num_pages, page_size, num_kv_heads, head_dim,
                                   kv_dtype, float(k_scale), float(v_scale), _ptr(k_pool),
                                   _ptr(v_pool)))


def attention(q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_pages, page_size,
              num_kv_heads, head_dim, kv_dtype, k_scale, v_scale, k_pool, v_pool,
              softmax_scale=0.0, n_threads=1) -> np.ndarray:
    """Exact attention of each row over its sequence's keys 0..position, in FP64.

    Returns float64 ``[n_rows][num_q_heads][head_dim]``.
    """
    q = np.ascontiguousarray(q)
    assert q.dtype == _NP_OF[q_dtype]
    seq_ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    n = int(seq_ids.shape[0])
    num_seqs, max_blocks = block_tables.shape
    out = np.zeros((n, num_q_heads, head_dim), dtype=np.float64)
    if np.ndim(k_scale) or np.ndim(v_scale):  # one scale per kv head
        ks, vs = _head_scales(k_scale, num_kv_heads), _head_scales(v_scale, num_kv_heads)
        st = lib().oracle_attention_h(n, _ptr(q), q_dtype, num_q_heads, _ptr(seq_ids), _ptr(positions),
                                      _ptr(block_tables), num_seqs, max_blocks, num_pages, page_size,
                                      num_kv_heads, head_dim, kv_dtype, _ptr(ks), _ptr(vs),
                                      _ptr(np.ascontiguousarray(k_pool)), _ptr(np.ascontiguousarray(v_pool)),
                                      float(softmax_scale), _ptr(out), int(n_threads))
    else:
        st = lib().oracle_attention(n, _ptr(q), q_dtype, num_q_heads, _ptr(seq_ids), _ptr(positions),
                                    _ptr(block_tables), num_seqs, max_blocks, num_pages, page_size,
                                    num_kv_heads, head_dim, kv_dtype, float(k_scale), float(v_scale),
                                    _ptr(np.ascontiguousarray(k_pool)), _ptr(np.ascontiguousarray(v_pool)),
                                    float(softmax_scale), _ptr(out), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attention failed with status {st}")
    return out


def workload_pools(wl, rows_of_seqs=None, include_step=True):
    """The oracle's own pools for a synthetic workload (any object with the
    fields of workloads.Workload): its append of the history rows (optionally
    only those that write pages of some sequences), then of the step's rows.
    Returns (k_pool, v_pool), poisoned where nothing was written."""
    kp, vp = wl.empty_pool(), wl.empty_pool()
    hs, hp, hk, hv = wl.hist_seq, wl.hist_pos, wl.hist_k, wl.hist_v
    if rows_of_seqs is not None:
        # pages of the chosen sequences may be shared with others (a shared
        # prefix): keep every history row that writes one of their pages
        pages = set(int(x) for x in wl.block_tables[list(rows_of_seqs)].reshape(-1) if x >= 0)
        tgt = wl.block_tables[hs, hp // wl.P]
        sel = np.isin(tgt, list(pages))
        hs, hp, hk, hv = hs[sel], hp[sel], hk[sel], hv[sel]
    st = append(hk, hv, wl.in_dtype, hs, hp, wl.block_tables, wl.num_pages, wl.P, wl.Hkv, wl.D,
                wl.kv_dtype, wl.k_scale, wl.v_scale, kp, vp)
    if st != 0:
        raise ValueError(f"oracle_append (history) failed with status {st}")
    if include_step:
        st = append(wl.k_new, wl.v_new, wl.in_dtype, wl.seq_ids, wl.positions, wl.block_tables,
                    wl.num_pages, wl.P, wl.Hkv, wl.D, wl.kv_dtype, wl.k_scale, wl.v_scale, kp, vp)
        if st != 0:
            raise ValueError(f"oracle_append (step) failed with status {st}")
    return kp, vp


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
