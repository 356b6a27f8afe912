"""pa_step (append + attention, the attention launched as a programmatic
dependent of the append) against the two separate calls: pool bytes and
outputs bit-identical, on every small workload (SIMT units, tensor-core e4m3
units, the mixed decode + prefill-tile launch), inside a captured CUDA graph,
and with the attention's start-up overlapping a long append."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def two_calls(wl):
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return st


def one_call(wl):
    st = pa_setup.upload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return st


def same(a, b):
    """Byte equality (the pools hold NaN-poisoned slots, which == would reject)."""
    for x, y in ((a.k_pool, b.k_pool), (a.v_pool, b.v_pool), (a.out, b.out)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("name", list(W.SMALL))
def test_step_matches_append_then_attention(name):
    same(two_calls(W.SMALL[name]()), one_call(W.SMALL[name]()))


def test_step_in_a_cuda_graph():
    wl = W.SMALL["mixed_step"]()
    ref = two_calls(wl)
    st = pa_setup.upload(wl)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        st.step(stream=s)  # first call outside capture (encodes the tensor maps)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            st.step(stream=s)
    torch.cuda.synchronize()
    for _ in range(3):
        st.out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    same(ref, st)


def test_step_after_a_long_append():
    """Many rows appended in the step itself (a whole prompt chunk per sequence):
    the dependent attention must see every appended row."""
    wl = W.chunked_step(61, chunks=[(0, 700, 704), (100, 300, 416)], decode_ctx=[40, 900])
    same(two_calls(wl), one_call(wl))


def _as_f32_inputs(wl):
    """The same workload with its appended rows given as f32 (the bf16 values,
    exactly), so the append converts f32 -> pool dtype."""
    for name in ("hist_k", "hist_v", "k_new", "v_new"):
        setattr(wl, name, W.as_f32(getattr(wl, name), wl.in_dtype))
    wl.in_dtype = W.F32
    return wl


def _fp8(wl, ks=0.0173, vs=0.0119):
    wl.k_scale, wl.v_scale = ks, vs
    return wl


CASES = {
    # f32 rows into bf16 and e4m3 pools: the units' own append converts like the append kernel
    "f32_in_bf16_pool_g2": lambda: _as_f32_inputs(W.batched_decode(n_seqs=12)),
    "f32_in_bf16_pool_g4": lambda: _as_f32_inputs(W.long_context(n_seqs=2, ctx=700)),
    "f32_in_e4m3_pool_g7": lambda: _as_f32_inputs(W.shared_prefix(n_seqs=24)),
    # head_dim 64 (two elements a lane), SIMT units, bf16 and e4m3 pools
    "d64_bf16": lambda: W._decode_workload("d64", 81, [1, 33, 300, 777], 8, 2, 64, 32, W.BF16, W.BF16, max_ctx=800,
                                           spare_pages=3, description="d64 bf16"),
    "d64_e4m3": lambda: _fp8(W._decode_workload("d64e", 82, [1, 33, 300, 777], 8, 2, 64, 32, W.E4M3, W.BF16,
                                                max_ctx=800, spare_pages=3, description="d64 e4m3")),
    # f32 queries on an e4m3 pool take the SIMT units
    "e4m3_f32q": lambda: _fp8(W._decode_workload("f32q", 83, [2, 65, 400], 14, 2, 128, 32, W.E4M3, W.F32,
                                                 max_ctx=448, spare_pages=3, description="e4m3 f32 q")),
    # pages of 16 and 256 tokens on every unit kind
    "p16_g2": lambda: W._decode_workload("p16", 84, [1, 16, 17, 513], 16, 8, 128, 16, W.BF16, W.BF16, max_ctx=528,
                                         spare_pages=3, description="p16"),
    "p256_g4": lambda: W._decode_workload("p256", 85, [1, 255, 256, 257, 900], 32, 8, 128, 256, W.BF16, W.BF16,
                                          max_ctx=1024, spare_pages=3, description="p256"),
    "p256_e4m3_g7": lambda: _fp8(W._decode_workload("p256e", 86, [1, 255, 257, 600], 28, 4, 128, 256, W.E4M3,
                                                    W.BF16, max_ctx=768, spare_pages=3, description="p256 e4m3")),
    # a short chunk (decode path, appended by the chunk append) beside rows that append themselves
    "short_chunk_beside_decode_rows": lambda: W.chunked_step(62, chunks=[(100, 8, 120), (40, 300, 352)],
                                                             decode_ctx=[5, 64, 900]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_matches_append_then_attention_more_shapes(name):
    same(two_calls(CASES[name]()), one_call(CASES[name]()))


@pytest.mark.parametrize("split", [64, 256])
def test_step_with_many_splits(split):
    """Rows split into many key ranges: the last range's unit appends the row."""
    old = pa.get_split_tokens()
    pa.set_split_tokens(split)
    try:
        for name in ("batched_decode", "shared_prefix", "long_context"):
            same(two_calls(W.SMALL[name]()), one_call(W.SMALL[name]()))
    finally:
        pa.set_split_tokens(old)


def test_step_with_a_bad_page_matches_two_calls():
    """A decode row whose last page id is out of range: both forms skip its
    append, report PA_ERR_OUT_OF_RANGE, and leave the same pool bytes."""
    outs = []
    for one in (False, True):
        wl = W.SMALL["shared_prefix"]()
        wl.block_tables = wl.block_tables.copy()
        st = pa_setup.upload(wl)
        bt = st.block_tables.clone()
        last = int((wl.positions[3]) // wl.P)
        bt[int(wl.seq_ids[3]), last] = wl.num_pages + 5
        st.block_tables = bt
        st.status.zero_()
        if one:
            st.step()
        else:
            st.append_step()
            st.attend()
        torch.cuda.synchronize()
        assert int(st.status.item()) == pa.PA_ERR_OUT_OF_RANGE
        outs.append(st)
    for x, y in ((outs[0].k_pool, outs[1].k_pool), (outs[0].v_pool, outs[1].v_pool)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    keep = [i for i in range(outs[0].out.shape[0]) if i != 3]
    assert torch.equal(outs[0].out[keep].view(torch.int16), outs[1].out[keep].view(torch.int16))
