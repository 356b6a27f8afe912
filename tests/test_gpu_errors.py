"""Device-side failure detection without faulting the GPU: out-of-range ids
and bounded waits that run out are reported in the status word, the kernels
return normally, and the context stays usable."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step():
    wl = W.batched_decode(n_seqs=32)
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return st


def _run(st, seq_ids=None, positions=None, bt=None):
    out = torch.empty_like(st.q)
    st.status.zero_()
    pa.attention(st.pool, st.q, st.seq_ids if seq_ids is None else seq_ids,
                 st.positions if positions is None else positions,
                 st.block_tables if bt is None else bt, out, workspace=st.workspace, status=st.status)
    torch.cuda.synchronize()
    return int(st.status.item()), out


def test_bad_sequence_id_reports_and_zeroes_row(step):
    good = step.out.clone()
    seq = step.seq_ids.clone()
    seq[4] = 10_000
    code, out = _run(step, seq_ids=seq)
    assert code == pa.PA_ERR_OUT_OF_RANGE
    assert torch.count_nonzero(out[4].float()) == 0
    others = [i for i in range(step.wl.n_rows) if i != 4]
    assert torch.equal(out[others].view(torch.int16), good[others].view(torch.int16))


def test_bad_position_reports(step):
    pos = step.positions.clone()
    pos[0] = step.wl.max_blocks * step.wl.P  # one past the table
    code, _ = _run(step, positions=pos)
    assert code == pa.PA_ERR_OUT_OF_RANGE


def test_bad_page_id_reports(step):
    bt = step.block_tables.clone()
    bt[7, 0] = step.wl.num_pages + 5
    code, out = _run(step, bt=bt)
    assert code == pa.PA_ERR_OUT_OF_RANGE
    assert torch.equal(out[8:].view(torch.int16), step.out[8:].view(torch.int16))


def test_wait_limit_runs_out_cleanly_and_context_survives(step):
    """Every CTA waits on a barrier nothing completes (the library's injected
    stall): the bounded wait runs out, the call reports PA_ERR_TIMEOUT, and the
    next normal call on the same context gives the same bits as before."""
    good = step.out.clone()
    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        code, _ = _run(step)
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert code == pa.PA_ERR_TIMEOUT
    code, out = _run(step)
    assert code == 0
    assert torch.equal(out.view(torch.int16), good.view(torch.int16))


def test_append_bad_rows_reported_others_written():
    wl = W.tiny_decode()
    st = pa_setup.upload(wl)
    seq = st.seq_ids.clone()
    seq[1] = -1
    st.status.zero_()
    pa.append_kv(st.pool, st.k_new, st.v_new, seq, st.positions, st.block_tables, status=st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == pa.PA_ERR_OUT_OF_RANGE
    k = st.k_pool.cpu()
    for r in (0, 2, 3):
        s, p = int(wl.seq_ids[r]), int(wl.positions[r])
        page = int(wl.block_tables[s, p // wl.P])
        assert torch.equal(k[page, :, p % wl.P, :], st.k_new[r].cpu())
