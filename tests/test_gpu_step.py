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
