"""Decode rows launched longest first (pa_set_unit_order): the order moves
where a row's units run, never what they compute, so every output byte and
every pool byte must equal the call-order launch's, on every unit kind (SIMT
f32 / bf16 / e4m3, the bf16 and e4m3 tensor-core units, the mixed launch with
prefill tiles), for split rows, rows with errors, rows that append themselves
inside the launch (pa_step, alone and in a CUDA graph), and with the order
written by the step's append launch.  The order itself is a permutation of the
rows with non-increasing unit length; the automatic mode orders exactly the
calls it documents; row groups keep the call's order; and a timeout still
reaches the status word with the order launch in front."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def restore_settings():
    old = (pa.get_unit_order(), pa.get_row_groups(), pa.get_split_tokens())
    yield
    pa.set_unit_order(old[0])
    pa.set_row_groups(old[1])
    pa.set_split_tokens(old[2])


def u8(t):
    return t.reshape(-1).view(torch.uint8)


def run(wl, mode, step, bt=None, seq_ids=None, positions=None):
    """Upload, then one pa_step (step=True) or append + pa_attention under
    `mode`.  Returns (pool bytes, output bytes, status, launches of the call)."""
    pa.set_unit_order(mode)
    st = pa_setup.upload(wl)
    if bt is not None or seq_ids is not None or positions is not None:
        st.block_tables = st.block_tables if bt is None else bt
        st.seq_ids = st.seq_ids if seq_ids is None else seq_ids
        st.positions = st.positions if positions is None else positions
    if not step:
        st.append_step()
        torch.cuda.synchronize()
    st.status.zero_()
    n0 = pa.kernel_launches()
    (st.step if step else st.attend)()
    launches = pa.kernel_launches() - n0
    torch.cuda.synchronize()
    pools = torch.cat([u8(st.k_pool), u8(st.v_pool)])
    return pools, u8(st.out).clone(), int(st.status.item()), launches


def assert_same(a, b, what):
    assert a[2] == b[2], f"{what}: status {a[2]} against {b[2]}"
    assert torch.equal(a[0], b[0]), f"{what}: pool bytes differ"
    if not torch.equal(a[1], b[1]):
        bad = int((a[1] != b[1]).nonzero()[0])
        raise AssertionError(f"{what}: output bytes differ (first at byte {bad})")


def _fp8(wl, ks=0.0173, vs=0.0119):
    wl.k_scale, wl.v_scale = ks, vs
    return wl


CASES = {
    **{name: W.SMALL[name] for name in W.SMALL},
    "d64_bf16": lambda: W._decode_workload("d64", 81, [1, 33, 300, 777, 64, 5], 8, 2, 64, 32, W.BF16, W.BF16,
                                           max_ctx=800, spare_pages=3, description="d64 bf16"),
    "e4m3_f32q": lambda: _fp8(W._decode_workload("f32q", 83, [2, 65, 400, 31, 390], 14, 2, 128, 32, W.E4M3, W.F32,
                                                 max_ctx=448, spare_pages=3, description="e4m3 f32 q")),
    "p256_g4": lambda: W._decode_workload("p256", 85, [1, 255, 256, 257, 900], 32, 8, 128, 256, W.BF16, W.BF16,
                                          max_ctx=1024, spare_pages=3, description="p256"),
    "short_chunk_beside_decode_rows": lambda: W.chunked_step(62, chunks=[(100, 8, 120), (40, 300, 352)],
                                                             decode_ctx=[5, 64, 900, 700, 3]),
}


@pytest.mark.parametrize("step", [False, True], ids=["attention", "step"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_longest_first_changes_no_bits(name, step):
    a = run(CASES[name](), pa.PA_ORDER_CALL, step)
    b = run(CASES[name](), pa.PA_ORDER_LONGEST_FIRST, step)
    assert a[2] == 0
    assert_same(a, b, f"{name} {'step' if step else 'attention'}")
    # one launch more for the order, except in a step with chunks, whose append launch writes it
    assert b[3] == a[3] + (0 if step and CASES[name]().chunks else 1)


@pytest.mark.parametrize("split", [64, 256])
def test_split_rows_longest_first(split):
    """Units hold at most `split` keys: long rows and short ones tie on their
    longest unit; the merge of a row's splits is the same."""
    pa.set_split_tokens(split)
    for name in ("batched_decode", "long_context", "batched_decode_fp8"):
        assert_same(run(W.SMALL[name](), pa.PA_ORDER_CALL, True), run(W.SMALL[name](), pa.PA_ORDER_LONGEST_FIRST, True),
                    f"{name}, split {split}")


def _unit_key(pos, split):
    return -(-min(pos + 1, split) // 32)


def test_order_is_a_permutation_longest_first():
    wl = W.batched_decode(seed=21, n_seqs=300, ctx_lo=1, ctx_hi=1200)
    pa.set_unit_order(pa.PA_ORDER_LONGEST_FIRST)
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    # the order is the workspace's last region (after any split partials)
    order_bytes = (wl.n_rows * 4 + 255) // 256 * 256
    ws = st.workspace.view(torch.int32)
    order = ws[(st.workspace.numel() - order_bytes) // 4:][: wl.n_rows].cpu().numpy()
    assert sorted(order.tolist()) == list(range(wl.n_rows))
    keys = np.array([_unit_key(int(wl.positions[r]), pa.get_split_tokens()) for r in order])
    assert (np.diff(keys) <= 0).all()


def test_auto_mode_orders_the_calls_it_documents():
    """At least 128 decode rows whose units can hold 1024 keys: ordered (one
    launch more), against the oracle on sampled rows; fewer rows or short
    tables: the call's order, one launch."""
    pa.set_unit_order(pa.PA_ORDER_AUTO)
    wl = W.batched_decode(seed=22, n_seqs=160, ctx_lo=64, ctx_hi=1300)
    assert wl.max_blocks * wl.P >= 1024
    ordered = run(wl, pa.PA_ORDER_AUTO, False)
    plain = run(wl, pa.PA_ORDER_CALL, False)
    assert ordered[3] == 2 and plain[3] == 1
    assert_same(plain, ordered, "auto against call order")
    rows = np.arange(0, wl.n_rows, 7)
    kp, vp = oracle_pools(wl)
    bits = ordered[1].cpu().numpy().view(np.uint16).reshape(wl.n_rows, wl.Hq, wl.D)
    got = W.bf16_bits_to_f32(bits)[rows]
    assert_close(got.astype(np.float64), oracle_out(wl, kp, vp, rows=rows), wl, "auto order")
    for small in (W.batched_decode(seed=23, n_seqs=100, ctx_hi=1300), W.shared_prefix(n_seqs=200)):
        assert run(small, pa.PA_ORDER_AUTO, False)[3] == 1


def test_rows_with_errors_longest_first():
    """A row whose sequence id is past the table and a row whose position is
    past its block table go last; zeros and PA_ERR_OUT_OF_RANGE for them, the
    same bytes everywhere else."""
    wl = W.SMALL["batched_decode"]()
    seq = torch.from_numpy(wl.seq_ids.copy()).cuda()
    pos = torch.from_numpy(wl.positions.copy()).cuda()
    seq[4] = wl.num_seqs + 3
    pos[9] = wl.max_blocks * wl.P
    a = run(wl, pa.PA_ORDER_CALL, False, seq_ids=seq, positions=pos)
    b = run(W.SMALL["batched_decode"](), pa.PA_ORDER_LONGEST_FIRST, False, seq_ids=seq, positions=pos)
    assert a[2] == pa.PA_ERR_OUT_OF_RANGE
    assert_same(a, b, "rows with errors")


def test_step_with_order_in_a_cuda_graph():
    wl = W.SMALL["batched_decode_fp8"]()
    ref = run(wl, pa.PA_ORDER_CALL, True)
    pa.set_unit_order(pa.PA_ORDER_LONGEST_FIRST)
    st = pa_setup.upload(wl)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        st.step(stream=s)  # first call outside capture (encodes the tensor maps); appending again writes the same bytes
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            st.step(stream=s)
    torch.cuda.synchronize()
    for _ in range(3):
        st.out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    assert_same(ref, (torch.cat([u8(st.k_pool), u8(st.v_pool)]), u8(st.out), 0, 0), "graph replay")


def test_row_groups_keep_the_call_order():
    wl = W.group_by_prefix(W.shared_prefix(n_seqs=40))
    pa.set_row_groups(1)
    a = run(wl, pa.PA_ORDER_CALL, False)
    pa.set_row_groups(8)
    b = run(wl, pa.PA_ORDER_LONGEST_FIRST, False)
    assert b[3] == 1, "row groups launch no order"
    assert_same(a, b, "row groups with longest-first asked for")


def test_timeout_reported_with_the_order_in_front():
    wl = W.SMALL["batched_decode"]()
    good = run(wl, pa.PA_ORDER_LONGEST_FIRST, False)
    pa.set_unit_order(pa.PA_ORDER_LONGEST_FIRST)
    st = pa_setup.upload(wl)
    st.append_step()
    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        st.attend()
        torch.cuda.synchronize()
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert int(st.status.item()) == pa.PA_ERR_TIMEOUT
    if st.workspace is not None:
        st.workspace.zero_()
    st.status.zero_()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    assert torch.equal(u8(st.out), good[1])


def test_many_rows_in_several_passes():
    """More rows than the order CTA has threads, in both places the order is
    written: a launch of its own (1024 threads: 2500 rows) and the step's
    append launch (256 threads: 700 decode rows beside a chunk)."""
    rng = np.random.default_rng(5)
    many = W._decode_workload("many", 91, rng.integers(1, 200, size=2500).tolist(), 2, 1, 64, 16, W.BF16, W.BF16,
                              max_ctx=208, spare_pages=3, description="2500 short rows")
    assert_same(run(many, pa.PA_ORDER_CALL, False), run(many, pa.PA_ORDER_LONGEST_FIRST, False), "2500 rows")
    pa.set_unit_order(pa.PA_ORDER_LONGEST_FIRST)
    st = pa_setup.upload(many)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    order_bytes = (many.n_rows * 4 + 255) // 256 * 256
    order = st.workspace.view(torch.int32)[(st.workspace.numel() - order_bytes) // 4:][: many.n_rows].cpu().numpy()
    assert sorted(order.tolist()) == list(range(many.n_rows))
    keys = np.array([_unit_key(int(many.positions[r]), pa.get_split_tokens()) for r in order])
    assert (np.diff(keys) <= 0).all()
    mixed = W.chunked_step(63, chunks=[(300, 40, 352)], decode_ctx=rng.integers(1, 400, size=700).tolist(), Hq=4,
                           Hkv=2, D=64, P=16)
    a = run(mixed, pa.PA_ORDER_CALL, True)
    b = run(mixed, pa.PA_ORDER_LONGEST_FIRST, True)
    assert a[2] == 0 and b[3] == a[3], "the append launch carries the order: no extra launch"
    assert_same(a, b, "700 decode rows beside a chunk, pa_step")
