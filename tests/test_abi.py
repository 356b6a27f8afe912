"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/pa.h declares, and its host-side argument checks
return the documented status codes without launching anything."""
import ctypes

import pytest

import paged_kv_continuous_pa_gb300 as pa
from paged_kv_continuous_pa_gb300 import build as pa_build


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load()


def test_exports_every_declared_function(lib):
    names = pa.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/pa.h but not exported"


def test_no_oracle_symbols_in_library(lib):
    for n in ("oracle_attention", "oracle_append", "oracle_e4m3_from_f32"):
        with pytest.raises(AttributeError):
            getattr(lib, n)


def _desc(**kw):
    d = dict(num_pages=16, page_size=32, num_kv_heads=2, head_dim=64, kv_dtype=pa.PA_BF16, k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return pa.PoolDesc(**d)


def test_pool_bytes(lib):
    assert lib.pa_pool_bytes(ctypes.byref(_desc())) == 16 * 2 * 32 * 64 * 2
    assert lib.pa_pool_bytes(ctypes.byref(_desc(kv_dtype=pa.PA_FP8_E4M3, k_scale=0.1, v_scale=0.1))) == 16 * 2 * 32 * 64
    assert lib.pa_pool_bytes(ctypes.byref(_desc(kv_dtype=pa.PA_F32))) == 16 * 2 * 32 * 64 * 4
    assert lib.pa_pool_bytes(ctypes.byref(_desc(head_dim=96))) == 0
    assert lib.pa_pool_bytes(None) == 0


def _create(lib, desc, k=0x10000, v=0x20000):
    h = ctypes.c_void_p()
    st = lib.pa_pool_create(ctypes.byref(desc), ctypes.c_void_p(k), ctypes.c_void_p(v), ctypes.byref(h))
    return st, h


def test_pool_create_validation(lib):
    st, h = _create(lib, _desc())
    assert st == pa.PA_OK and h.value
    lib.pa_pool_destroy(h)
    assert _create(lib, _desc(head_dim=96))[0] == pa.PA_ERR_UNSUPPORTED
    assert _create(lib, _desc(page_size=8))[0] == pa.PA_ERR_UNSUPPORTED
    assert _create(lib, _desc(page_size=48))[0] == pa.PA_ERR_UNSUPPORTED  # not a power of two
    assert _create(lib, _desc(page_size=512))[0] == pa.PA_ERR_UNSUPPORTED
    for ps in (16, 32, 64, 128, 256):
        st, h = _create(lib, _desc(page_size=ps))
        assert st == pa.PA_OK
        lib.pa_pool_destroy(h)
    assert _create(lib, _desc(num_pages=0))[0] == pa.PA_ERR_INVALID_ARG
    assert _create(lib, _desc(kv_dtype=7))[0] == pa.PA_ERR_INVALID_ARG
    assert _create(lib, _desc(kv_dtype=pa.PA_FP8_E4M3, k_scale=0.0))[0] == pa.PA_ERR_INVALID_ARG
    assert _create(lib, _desc(kv_dtype=pa.PA_FP8_E4M3, v_scale=float("inf")))[0] == pa.PA_ERR_INVALID_ARG
    assert _create(lib, _desc(), k=0x10008)[0] == pa.PA_ERR_INVALID_ARG  # not 16-byte aligned
    assert _create(lib, _desc(), k=0)[0] == pa.PA_ERR_INVALID_ARG
    assert "aligned" in pa.last_error() or "NULL" in pa.last_error()


def test_host_side_errors_launch_nothing(lib):
    st, h = _create(lib, _desc())
    assert st == pa.PA_OK
    try:
        vp = ctypes.c_void_p
        dev = vp(0x100000)
        # bad input dtype
        assert lib.pa_append_kv(h, 4, dev, dev, pa.PA_FP8_E4M3, dev, dev, dev, 4, 4, None, None) == pa.PA_ERR_INVALID_ARG
        # zero rows is a no-op
        assert lib.pa_append_kv(h, 0, None, None, pa.PA_BF16, None, None, None, 4, 4, None, None) == pa.PA_OK
        # misaligned k_new
        assert lib.pa_append_kv(h, 4, vp(0x100004), dev, pa.PA_BF16, dev, dev, dev, 4, 4, None, None) == pa.PA_ERR_INVALID_ARG
        att = lambda **kw: lib.pa_attention(h, kw.get("n", 4), dev, kw.get("qd", pa.PA_BF16), kw.get("hq", 8), dev,
                                            dev, dev, 4, kw.get("mb", 4), kw.get("chunks"), kw.get("nc", 0), 0.0,
                                            kw.get("out", dev), kw.get("ws"), kw.get("wsb", 0), None, None)
        assert att(hq=5) == pa.PA_ERR_INVALID_ARG
        assert att(hq=18) == pa.PA_ERR_UNSUPPORTED         # group of 9
        assert att(qd=pa.PA_FP8_E4M3) == pa.PA_ERR_INVALID_ARG
        assert att(out=None) == pa.PA_ERR_INVALID_ARG
        assert att(out=vp(0x100008)) == pa.PA_ERR_INVALID_ARG   # out not 16-byte aligned
        assert lib.pa_attention(h, 4, vp(0x100002), pa.PA_BF16, 8, dev, dev, dev, 4, 4, None, 0, 0.0, dev, None, 0,
                                None, None) == pa.PA_ERR_INVALID_ARG  # q not 16-byte aligned
        assert att(n=0, out=None) == pa.PA_OK
        two = (pa.Chunk * 2)(pa.Chunk(0, 3), pa.Chunk(2, 2))
        assert att(chunks=two, nc=2) == pa.PA_ERR_INVALID_ARG   # overlapping chunks
        assert att(chunks=None, nc=1) == pa.PA_ERR_INVALID_ARG
        assert att(nc=17) == pa.PA_ERR_INVALID_ARG
        # pa_step checks every argument of both halves before launching anything: a bad
        # attention argument returns INVALID_ARG, not the CUDA error the append's launch
        # would give on this GPU-less machine
        stp = lambda **kw: lib.pa_step(h, 4, dev, pa.PA_BF16, kw.get("hq", 8), dev, dev, kw.get("ind", pa.PA_BF16), dev,
                                       dev, dev, 4, 4, None, 0, 0.0, kw.get("out", dev), None, 0, None, None)
        assert stp(ind=pa.PA_FP8_E4M3) == pa.PA_ERR_INVALID_ARG
        assert stp(hq=5) == pa.PA_ERR_INVALID_ARG
        assert stp(out=None) == pa.PA_ERR_INVALID_ARG
        assert stp(out=vp(0x100008)) == pa.PA_ERR_INVALID_ARG
        # long tables need a workspace for split partials
        need = lib.pa_attention_workspace_bytes(h, 4, 8, 200, None, 0)
        assert need > 0 and need % 256 == 0
        assert att(mb=200) == pa.PA_ERR_INVALID_ARG
        assert att(mb=200, ws=vp(0x200000), wsb=need - 1) == pa.PA_ERR_INVALID_ARG
        assert att(mb=200, ws=vp(0x200010), wsb=need) == pa.PA_ERR_INVALID_ARG  # not 256-aligned
        assert lib.pa_attention_workspace_bytes(h, 4, 8, 4, None, 0) == 0  # 128 tokens: never split
        one = (pa.Chunk * 1)(pa.Chunk(0, 4))
        assert lib.pa_attention_workspace_bytes(h, 4, 8, 4, one, 1) == 0  # chunk below the tile threshold
        big = (pa.Chunk * 1)(pa.Chunk(0, 64))
        # 6400 keys: tile key ranges split (4096 keys per range), on top of the decode splits
        assert lib.pa_attention_workspace_bytes(h, 64, 8, 200, big, 1) > lib.pa_attention_workspace_bytes(h, 64, 8, 200, None, 0)
    finally:
        lib.pa_pool_destroy(h)


def test_split_tokens_setting(lib):
    old = lib.pa_get_split_tokens()
    try:
        assert lib.pa_set_split_tokens(100) == pa.PA_ERR_INVALID_ARG
        assert lib.pa_set_split_tokens(0) == pa.PA_ERR_INVALID_ARG
        assert lib.pa_set_split_tokens(512) == pa.PA_OK and lib.pa_get_split_tokens() == 512
    finally:
        lib.pa_set_split_tokens(old)


def test_row_groups_setting(lib):
    old = lib.pa_get_row_groups()
    assert old == 1  # one row per CTA unless the caller asks
    try:
        for bad in (0, 3, 5, 16, -2):
            assert lib.pa_set_row_groups(bad) == pa.PA_ERR_INVALID_ARG
            assert lib.pa_get_row_groups() == old
        for rows in (2, 4, 8, 1):
            assert lib.pa_set_row_groups(rows) == pa.PA_OK and lib.pa_get_row_groups() == rows
    finally:
        lib.pa_set_row_groups(old)


def test_unit_order_setting(lib):
    old = lib.pa_get_unit_order()
    assert old == pa.PA_ORDER_AUTO
    st, h = _create(lib, _desc())  # P 32, 2 kv heads, D 64
    assert st == pa.PA_OK
    try:
        for bad in (-1, 3, 7):
            assert lib.pa_set_unit_order(bad) == pa.PA_ERR_INVALID_ARG
            assert lib.pa_get_unit_order() == old
        ws = lambda n, mb, chunks=None: lib.pa_attention_workspace_bytes(h, n, 8, mb, chunks, 1 if chunks else 0)
        # 40 pages of 32 tokens: units up to 1280 keys, never split; the order takes n_rows int32, padded to 256
        assert lib.pa_set_unit_order(pa.PA_ORDER_AUTO) == pa.PA_OK
        assert ws(200, 40) == 1024     # 200 rows: ordered
        assert ws(127, 40) == 0        # too few rows to order
        assert ws(200, 20) == 0        # units of at most 640 keys
        whole = (pa.Chunk * 1)(pa.Chunk(0, 200))
        assert ws(200, 40, whole) == 1024  # room kept although bf16 queries would run every row as a tile
        assert lib.pa_set_unit_order(pa.PA_ORDER_CALL) == pa.PA_OK and lib.pa_get_unit_order() == pa.PA_ORDER_CALL
        assert ws(200, 40) == 0
        assert lib.pa_set_unit_order(pa.PA_ORDER_LONGEST_FIRST) == pa.PA_OK
        assert ws(100, 20) == 512 and ws(1, 20) == 0
    finally:
        lib.pa_set_unit_order(old)
        lib.pa_pool_destroy(h)


def test_settings_change_from_other_threads(lib):
    """One thread flips the split length while others size workspaces: every
    answer is the one of the two settings, never a mix (a call reads it once)."""
    import threading
    st, h = _create(lib, _desc())
    assert st == pa.PA_OK
    old = lib.pa_get_split_tokens()
    try:
        sizes = {}
        for t in (1024, 4096):
            assert lib.pa_set_split_tokens(t) == pa.PA_OK
            sizes[t] = lib.pa_attention_workspace_bytes(h, 64, 8, 200, None, 0)
        assert sizes[1024] > sizes[4096] > 0
        stop = threading.Event()
        seen, bad = set(), []

        def flip():
            i = 0
            while not stop.is_set():
                lib.pa_set_split_tokens((1024, 4096)[i % 2])
                i += 1

        def size():
            for _ in range(20000):
                v = lib.pa_attention_workspace_bytes(h, 64, 8, 200, None, 0)
                seen.add(v)
                if v not in sizes.values():
                    bad.append(v)

        threads = [threading.Thread(target=flip)] + [threading.Thread(target=size) for _ in range(3)]
        for t in threads:
            t.start()
        for t in threads[1:]:
            t.join()
        stop.set()
        threads[0].join()
        assert not bad and seen <= set(sizes.values())
    finally:
        lib.pa_set_split_tokens(old)
        lib.pa_pool_destroy(h)


def test_head_scales_validation(lib):
    arr = lambda *v: (ctypes.c_float * len(v))(*v)
    st, h = _create(lib, _desc(kv_dtype=pa.PA_FP8_E4M3, k_scale=0.5, v_scale=0.5))
    assert st == pa.PA_OK
    try:
        assert lib.pa_pool_set_head_scales(h, arr(0.1, 0.2), arr(0.3, 0.4)) == pa.PA_OK
        assert lib.pa_pool_set_head_scales(h, None, None) == pa.PA_OK  # back to per tensor
        assert lib.pa_pool_set_head_scales(h, arr(0.1, 0.2), None) == pa.PA_ERR_INVALID_ARG
        assert lib.pa_pool_set_head_scales(h, arr(0.1, 0.0), arr(0.3, 0.4)) == pa.PA_ERR_INVALID_ARG
        assert lib.pa_pool_set_head_scales(h, arr(0.1, 0.2), arr(float("nan"), 0.4)) == pa.PA_ERR_INVALID_ARG
    finally:
        lib.pa_pool_destroy(h)
    st, h = _create(lib, _desc())  # bf16
    assert lib.pa_pool_set_head_scales(h, arr(0.1, 0.2), arr(0.3, 0.4)) == pa.PA_ERR_INVALID_ARG
    lib.pa_pool_destroy(h)
    st, h = _create(lib, _desc(kv_dtype=pa.PA_FP8_E4M3, num_kv_heads=65))
    many = (ctypes.c_float * 65)(*([0.5] * 65))
    assert lib.pa_pool_set_head_scales(h, many, many) == pa.PA_ERR_UNSUPPORTED
    lib.pa_pool_destroy(h)


def test_status_strings(lib):
    for code, name in enumerate(["PA_OK", "PA_ERR_INVALID_ARG", "PA_ERR_UNSUPPORTED", "PA_ERR_OUT_OF_RANGE",
                                 "PA_ERR_TIMEOUT", "PA_ERR_CUDA", "PA_ERR_NO_PAGES"]):
        assert pa.status_string(code) == name


def test_noalloc_checks_arguments_then_its_scratch_size(lib):
    """pa_attention_noalloc checks its arguments as pa_attention does before it
    sizes its plan: a chunk of no rows is an invalid argument (not an
    unsupported size), and a plan beyond the 32 MiB scratch is refused before
    any CUDA call."""
    st, h = _create(lib, _desc(head_dim=128, num_kv_heads=8))
    assert st == pa.PA_OK
    try:
        dev = ctypes.c_void_p(0x100000)
        bad = (pa.Chunk * 1)(pa.Chunk(0, 0))
        assert lib.pa_attention_noalloc(h, 4, dev, pa.PA_BF16, 16, dev, dev, dev, 4, 2048, bad, 1, 0.0, dev, None,
                                        None) == pa.PA_ERR_INVALID_ARG
        assert "chunk" in pa.last_error()
        # 4096 rows x 64 splits of 16 heads: far more than 32 MiB of partials
        assert lib.pa_attention_noalloc(h, 4096, dev, pa.PA_BF16, 16, dev, dev, dev, 4096, 2048, None, 0, 0.0, dev,
                                        None, None) == pa.PA_ERR_UNSUPPORTED
        assert "scratch" in pa.last_error()
    finally:
        lib.pa_pool_destroy(h)
