"""Row groups of the e4m3 tensor-core decode units (pa_set_row_groups): one
CTA runs 2, 4 or 8 consecutive rows and copies the leading pages they all
share once.  Every output bit must equal the one-row-per-CTA units' (the
per-row arithmetic is the same), whatever the grouping, the page size, the
query-head group, the split length, the rows' order, and whether a row
appends its own key inside the launch; errors and timeouts are reported as
before and leave nothing behind for the next call."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu

ROW_GROUPS = (2, 4, 8)


@pytest.fixture(autouse=True)
def restore_settings():
    old_rg, old_split = pa.get_row_groups(), pa.get_split_tokens()
    yield
    pa.set_row_groups(old_rg)
    pa.set_split_tokens(old_split)


def attend(st, rows, bt=None, seq_ids=None):
    pa.set_row_groups(rows)
    out = torch.empty_like(st.q)
    st.status.zero_()
    pa.attention(st.pool, st.q, st.seq_ids if seq_ids is None else seq_ids, st.positions,
                 st.block_tables if bt is None else bt, out, softmax_scale=st.wl.softmax_scale,
                 workspace=st.workspace, status=st.status)
    torch.cuda.synchronize()
    return out, int(st.status.item())


def uploaded(wl):
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return st


def assert_bits_equal(a, b, what):
    a16, b16 = a.view(torch.int16), b.view(torch.int16)
    if not torch.equal(a16, b16):
        bad = (a16 != b16).reshape(a.shape[0], -1).any(dim=1).nonzero().flatten().tolist()
        raise AssertionError(f"{what}: rows {bad[:10]} differ from one row per CTA")


def check_groups_identical(wl, what):
    st = uploaded(wl)
    base, s0 = attend(st, 1)
    assert s0 == 0
    for rg in ROW_GROUPS:
        out, s = attend(st, rg)
        assert s == 0, f"{what}: status {s} with {rg} rows per CTA"
        assert_bits_equal(out, base, f"{what}, {rg} rows per CTA")
    return st, base


SHAPES = [  # (P, Hq, Hkv, prefix, prompt): G = Hq / Hkv
    (32, 28, 4, 90, 128),   # the shared-prefix shape: G 7, two shared pages
    (16, 8, 2, 90, 128),    # G 4 (hi and lo weights in one MMA), two pages per stage, five shared pages
    (64, 2, 2, 90, 128),    # G 1, one shared page = two stages
    (128, 16, 2, 300, 400),  # G 8, two shared pages of four stages each
]


@pytest.mark.parametrize("grouped", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"P{s[0]}-G{s[1] // s[2]}")
def test_bit_identical_to_one_row_per_cta(shape, grouped):
    P, Hq, Hkv, prefix, prompt = shape
    wl = W.shared_prefix(seed=40 + P, n_seqs=37, P=P, Hq=Hq, Hkv=Hkv, prefix=prefix, prompt=prompt)
    if grouped:
        wl = W.group_by_prefix(wl)
    check_groups_identical(wl, f"P{P} G{Hq // Hkv} {'grouped' if grouped else 'as drawn'}")


def test_against_the_oracle():
    wl = W.group_by_prefix(W.shared_prefix(n_seqs=40))
    st = uploaded(wl)
    out, s = attend(st, 8)
    assert s == 0
    kp, vp = oracle_pools(wl)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, "8 rows per CTA")


@pytest.mark.parametrize("split", [64, 256])
def test_split_rows(split):
    """Splits of 64 and 256 tokens: every split of a group computes its shared
    stages afresh (the leading pages of that key range)."""
    pa.set_split_tokens(split)
    wl = W.group_by_prefix(W.shared_prefix(seed=9, n_seqs=40, prefix=200, prompt=300, max_gen=300))
    check_groups_identical(wl, f"split {split}")


def test_rows_in_any_order_and_count():
    """Shuffled rows (groups that share only in part), a row count that is
    not a multiple of the group size, and one row alone."""
    wl = W.group_by_prefix(W.shared_prefix(seed=11, n_seqs=45))
    st = uploaded(wl)
    base, _ = attend(st, 1)
    rng = np.random.default_rng(3)
    for rows in (rng.permutation(wl.n_rows), np.arange(29), np.array([5]), np.r_[np.arange(8), np.arange(8)]):
        idx = torch.as_tensor(rows, dtype=torch.long, device="cuda")
        q = st.q[idx].contiguous()
        for rg in ROW_GROUPS:
            pa.set_row_groups(rg)
            out = torch.empty_like(q)
            st.status.zero_()
            pa.attention(st.pool, q, st.seq_ids[idx].contiguous(), st.positions[idx].contiguous(), st.block_tables,
                         out, softmax_scale=wl.softmax_scale, workspace=st.workspace, status=st.status)
            torch.cuda.synchronize()
            assert int(st.status.item()) == 0
            assert_bits_equal(out, base[idx], f"{len(rows)} rows, {rg} per CTA")


@pytest.mark.parametrize("rg", ROW_GROUPS)
def test_step_appends_inside_groups(rg):
    """pa_step with row groups: each row stores its own key and value inside
    the launch and patches its last stage; pool bytes and outputs equal the
    append + attention calls with one row per CTA."""
    wl = W.group_by_prefix(W.shared_prefix(seed=13, n_seqs=40))
    a = pa_setup.upload(wl)
    pa.set_row_groups(1)
    a.append_step()
    a.attend()
    b = pa_setup.upload(wl)
    pa.set_row_groups(rg)
    b.step()
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert_bits_equal(b.out, a.out, f"pa_step, {rg} rows per CTA")


def test_errors_inside_a_group():
    """A row with a page id past the pool and a row with a sequence id past the
    table, both inside groups of sharing rows: zeros and PA_ERR_OUT_OF_RANGE
    for them, the other rows' bits unchanged; then an injected stall times
    out, and the next call is exact again."""
    wl = W.group_by_prefix(W.shared_prefix(seed=17, n_seqs=40))
    st = uploaded(wl)
    good, _ = attend(st, 1)
    bt = st.block_tables.clone()
    bad_row, oob_row = 3, 10
    bt[int(wl.seq_ids[bad_row]), 0] = wl.num_pages + 1
    seq = st.seq_ids.clone()
    seq[oob_row] = wl.num_seqs
    for rg in ROW_GROUPS:
        out, s = attend(st, rg, bt=bt, seq_ids=seq)
        assert s == pa.PA_ERR_OUT_OF_RANGE
        for r in (bad_row, oob_row):
            assert torch.count_nonzero(out[r].float()) == 0
        keep = [i for i in range(wl.n_rows) if i not in (bad_row, oob_row)]
        assert_bits_equal(out[keep], good[keep], f"rows beside the errors, {rg} per CTA")

    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        _, s = attend(st, 8)
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert s == pa.PA_ERR_TIMEOUT
    out, s = attend(st, 8)
    assert s == 0
    assert_bits_equal(out, good, "after a timeout")
