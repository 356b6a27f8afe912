"""pa_attention_noalloc: attention for callers that cannot allocate device
memory (they are handed only input and output buffers, for instance by a
host runtime that owns all device memory, or may not call cudaMalloc on the
serving path).  Its split-KV scratch is a fixed 32 MiB array inside the
library.

Both entry points run the same kernels on the same plan, so their outputs must
be byte-identical: a tolerance would hide partials or counters left over in the
shared array by an earlier call.  Checked through the C ABI against
pa_attention (which takes a caller workspace) on two calls in a row, the
second with a different batch, and against the oracle; and through the Python
binding on a step whose chunk's key range is split across CTAs, so that the
tile path's partials and counters go through the shared array too."""
import ctypes

import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from paged_kv_continuous_pa_gb300 import build as pa_build
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


def _noalloc_raw(lib, st, q, seq, pos, out):
    """Call the C entry point directly with raw pointers."""
    num_seqs, max_blocks = (int(x) for x in st.block_tables.shape)
    return lib.pa_attention_noalloc(st.pool.handle, int(seq.shape[0]), q.data_ptr(), pa.PA_BF16, int(q.shape[1]),
                                    seq.data_ptr(), pos.data_ptr(), st.block_tables.data_ptr(), num_seqs, max_blocks,
                                    None, 0, 0.0, out.data_ptr(), st.status.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().tobytes()


def _with_split(tokens, fn):
    old = pa.get_split_tokens()
    pa.set_split_tokens(tokens)
    try:
        fn()
    finally:
        pa.set_split_tokens(old)


def test_noalloc_matches_workspace_entry_point_twice():
    pa_build.build()
    _with_split(1024, lambda: _compare_twice(pa.load()))  # rows longer than 1024 keys are split


def _compare_twice(lib):
    wl = W.batched_decode(n_seqs=40, ctx_lo=900)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    assert pa.workspace_bytes(st.pool, wl.n_rows, wl.Hq, wl.max_blocks) > 0
    kp, vp = oracle_pools(wl)

    batches = [np.arange(wl.n_rows), np.random.default_rng(1).permutation(wl.n_rows)[:29]]
    for call, rows in enumerate(batches):
        idx = torch.as_tensor(rows, dtype=torch.long, device="cuda")
        q = st.q[idx].contiguous()
        seq = st.seq_ids[idx].contiguous()
        pos = st.positions[idx].contiguous()
        ws_bytes = pa.workspace_bytes(st.pool, len(rows), wl.Hq, wl.max_blocks)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        ref_out = torch.empty_like(q)
        pa.attention(st.pool, q, seq, pos, st.block_tables, ref_out, workspace=ws, status=st.status)
        out = torch.full_like(q, float("nan"))
        st.status.zero_()
        assert _noalloc_raw(lib, st, q, seq, pos, out) == pa.PA_OK, pa.last_error()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        assert _bits(out) == _bits(ref_out), f"noalloc call {call + 1}: output bytes differ from pa_attention"
        if call == 0:
            got = W.bf16_bits_to_f32(pa_setup.to_numpy(out)).astype(np.float64)
            assert_close(got, oracle_out(wl, kp, vp, rows=rows), wl, "noalloc against the oracle")


def test_noalloc_tile_splits_through_the_binding_twice():
    """A bf16 step whose 64-row chunk reads 4264 keys (its key range is split
    across two CTAs per tile, more than 4096 keys) beside decode rows split at
    1024 keys: both kinds of partials and counters use the shared array."""
    pa_build.build()
    _with_split(1024, _tile_case)


def _tile_case():
    wl = W.chunked_step(61, chunks=[(4200, 64, 4300)], decode_ctx=[3000, 5000, 17])
    assert wl.max_blocks * wl.P > 4096
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    kp, vp = oracle_pools(wl)
    ref_out = torch.empty_like(st.q)
    ws_bytes = pa.workspace_bytes(st.pool, wl.n_rows, wl.Hq, wl.max_blocks, wl.chunks)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    pa.attention(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, ref_out, chunks=wl.chunks, workspace=ws,
                 status=st.status)
    for call in range(2):
        out = torch.full_like(st.q, float("nan"))
        st.status.zero_()
        pa.attention_noalloc(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, out, chunks=wl.chunks,
                             status=st.status)
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        assert _bits(out) == _bits(ref_out), f"noalloc call {call + 1}: output bytes differ from pa_attention"
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, "noalloc tile splits against the oracle")


def test_noalloc_rejects_calls_beyond_its_scratch():
    pa_build.build()
    lib = pa.load()
    k = torch.empty((8, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
    pool = pa.Pool(k, torch.empty_like(k))
    n, hq, mb = 4096, 16, 2048  # 64 splits per row: far more than 32 MiB of partials
    assert pa.workspace_bytes(pool, n, hq, mb) > 32 << 20
    dev = ctypes.c_void_p(k.data_ptr())
    st = lib.pa_attention_noalloc(pool.handle, n, dev, pa.PA_BF16, hq, dev, dev, dev, n, mb, None, 0, 0.0, dev,
                                  None, None)
    assert st == pa.PA_ERR_UNSUPPORTED
    assert "scratch" in pa.last_error()



def test_noalloc_with_rows_longest_first():
    """The decode rows' launch order (pa_set_unit_order) goes through the
    shared array too: bytes equal to pa_attention's in both orders, twice."""
    pa_build.build()
    old = pa.get_unit_order()
    wl = W.batched_decode(seed=31, n_seqs=48, ctx_lo=1, ctx_hi=1500)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    try:
        outs = []
        for mode in (pa.PA_ORDER_LONGEST_FIRST, pa.PA_ORDER_CALL, pa.PA_ORDER_LONGEST_FIRST):
            pa.set_unit_order(mode)
            ws = torch.zeros(max(pa.workspace_bytes(st.pool, wl.n_rows, wl.Hq, wl.max_blocks), 256), dtype=torch.uint8,
                             device="cuda")
            ref_out = torch.empty_like(st.q)
            pa.attention(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, ref_out, workspace=ws,
                         status=st.status)
            out = torch.full_like(st.q, float("nan"))
            pa.attention_noalloc(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, out, status=st.status)
            torch.cuda.synchronize()
            assert int(st.status.item()) == 0
            assert _bits(out) == _bits(ref_out), f"order mode {mode}: output bytes differ from pa_attention"
            outs.append(_bits(out))
        assert outs[0] == outs[1] == outs[2]
    finally:
        pa.set_unit_order(old)
