"""pa_attention_noalloc: attention for callers that cannot allocate device
memory (they are handed only input and output buffers, for instance by a
host runtime that owns all device memory, or may not call cudaMalloc on the
serving path).  Its split-KV scratch is a fixed 32 MiB array inside the
library.  Checked through the C ABI against pa_attention, which takes a
caller workspace, on two calls in a row (the second with a different batch,
so leftovers of the first call in the shared array would show)."""
import ctypes

import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from paged_kv_continuous_pa_gb300 import build as pa_build
from ref import assert_close

pytestmark = pytest.mark.gpu


def _noalloc_raw(lib, st, q, seq, pos, out):
    """Call the C entry point directly with raw pointers."""
    num_seqs, max_blocks = (int(x) for x in st.block_tables.shape)
    return lib.pa_attention_noalloc(st.pool.handle, int(seq.shape[0]), q.data_ptr(), pa.PA_BF16, int(q.shape[1]),
                                    seq.data_ptr(), pos.data_ptr(), st.block_tables.data_ptr(), num_seqs, max_blocks,
                                    None, 0, 0.0, out.data_ptr(), st.status.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice():
    pa_build.build()
    lib = pa.load()
    old_split = pa.get_split_tokens()
    pa.set_split_tokens(1024)  # so that the rows are split and the scratch is used
    try:
        _compare_twice(lib)
    finally:
        pa.set_split_tokens(old_split)


def _compare_twice(lib):
    wl = W.batched_decode(n_seqs=40, ctx_lo=900)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    assert pa.workspace_bytes(st.pool, wl.n_rows, wl.Hq, wl.max_blocks) > 0

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
        got = W.bf16_bits_to_f32(pa_setup.to_numpy(out)).astype(np.float64)
        ref = W.bf16_bits_to_f32(pa_setup.to_numpy(ref_out)).astype(np.float64)
        assert_close(got, ref, wl, f"noalloc call {call + 1}")


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
    assert "32" in pa.last_error() or "scratch" in pa.last_error()
