"""The tensor-core prefill-chunk tile path (tcgen05) against the oracle:
chunk lengths that leave ragged tiles, chunks starting at position 0, keys
past the chunk's last row on poisoned slots, several chunks and decode rows in
one launch, every group size, both head dims and all page sizes."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


def run_and_check(wl, what):
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    kp, vp = oracle_pools(wl)
    ref = oracle_out(wl, kp, vp)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    return assert_close(got, ref, wl, what)


@pytest.mark.parametrize("chunk", [(0, 16, 16), (0, 130, 150), (37, 64, 200), (100, 300, 420), (64, 257, 321)])
def test_single_chunk_shapes(chunk):
    run_and_check(W.chunked_step(11, [chunk]), f"chunk {chunk}")


@pytest.mark.parametrize("G", [1, 3, 4, 5, 8])
def test_group_sizes(G):
    run_and_check(W.chunked_step(20 + G, [(50, 140, 200)], decode_ctx=[70, 500], Hq=2 * G, Hkv=2), f"G{G}")


@pytest.mark.parametrize("D,P", [(64, 16), (64, 64), (128, 16), (128, 64), (128, 128), (64, 256)])
def test_head_dims_and_pages(D, P):
    run_and_check(W.chunked_step(30 + D + P, [(33, 97, 180)], decode_ctx=[5, 300], Hq=8, Hkv=2, D=D, P=P),
                  f"D{D} P{P}")


@pytest.mark.parametrize("P", [16, 32, 128, 256])
def test_long_tile_key_ranges_split_and_merge(P):
    """A chunk far into its sequence: each tile's keys span several key ranges
    that separate CTAs process and the last one merges in ascending order (at
    P = 16 a range's page-id table is at its largest, 256 pages)."""
    wl = W.chunked_step(45, [(9000, 200, 9300)], decode_ctx=[50, 7000], Hq=8, Hkv=2, P=P)
    run_and_check(wl, f"chunk at 9000, P{P}")


def test_sixteen_chunks_the_most_one_call_takes():
    """16 chunks in one launch (the limit), tile-path and decode-path chunks
    (one shorter than a tile's 16 rows) beside decode rows."""
    chunks = []
    for i in range(16):
        n = 5 if i == 6 else 16 + (i % 3) * 9
        start = 11 * i
        chunks.append((start, n, start + n + 7))
    run_and_check(W.chunked_step(61, chunks, decode_ctx=[3, 200, 650], Hq=8, Hkv=2), "16 chunks")


def test_several_chunks_with_decode_rows():
    wl = W.chunked_step(41, [(0, 40, 40), (200, 77, 300), (513, 128, 700)], decode_ctx=[1, 64, 999, 2000])
    run_and_check(wl, "three chunks + decode rows")


def test_chunk_rows_bit_identical_across_calls_and_batches():
    wl = W.chunked_step(51, [(300, 200, 600)], decode_ctx=[10, 400, 900])
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    first = st.out.view(torch.int16).clone()
    for _ in range(5):
        st.attend()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), first)
    # the chunk alone (no decode rows in the launch) gives the same chunk bits
    b, n = wl.chunks[0]
    sl = slice(b, b + n)
    out = torch.empty_like(st.q[sl])
    wsb = pa.workspace_bytes(st.pool, n, wl.Hq, wl.max_blocks, [(0, n)])
    ws = torch.zeros(max(wsb, 1), dtype=torch.uint8, device="cuda")
    pa.attention(st.pool, st.q[sl].contiguous(), st.seq_ids[sl].contiguous(), st.positions[sl].contiguous(),
                 st.block_tables, out, chunks=[(0, n)], workspace=ws, status=st.status)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), first[sl])


def test_short_chunk_and_f32_queries_use_the_decode_path():
    # 15 rows is below the tile threshold; f32 q cannot use the bf16 tensor cores
    run_and_check(W.chunked_step(61, [(20, 15, 40)], decode_ctx=[30]), "short chunk")
    wl = W.chunked_step(62, [(20, 90, 200)], decode_ctx=[30], q_dtype=W.F32, kv_dtype=W.F32)
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    kp, vp = oracle_pools(wl)
    assert_close(pa_setup.to_numpy(st.out).astype(np.float64), oracle_out(wl, kp, vp), wl, "f32 chunk")


def test_tile_path_timeout_reports_and_recovers():
    wl = W.chunked_step(71, [(500, 256, 800)], decode_ctx=[100, 2000])
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    good = st.out.view(torch.int16).clone()
    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        st.status.zero_()
        st.attend()
        torch.cuda.synchronize()
        code = int(st.status.item())
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert code == pa.PA_ERR_TIMEOUT
    st.status.zero_()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    assert torch.equal(st.out.view(torch.int16), good)


def chunk_alone(st, wl, c=0):
    """Chunk c of the workload attended in a call of its own (only tile-path
    rows: the launch of tile CTAs alone)."""
    b, n = wl.chunks[c]
    sl = slice(b, b + n)
    out = torch.empty_like(st.q[sl])
    wsb = pa.workspace_bytes(st.pool, n, wl.Hq, wl.max_blocks, [(0, n)])
    ws = torch.zeros(max(wsb, 1), dtype=torch.uint8, device="cuda")
    st.status.zero_()
    pa.attention(st.pool, st.q[sl].contiguous(), st.seq_ids[sl].contiguous(), st.positions[sl].contiguous(),
                 st.block_tables, out, chunks=[(0, n)], softmax_scale=wl.softmax_scale, workspace=ws, status=st.status)
    torch.cuda.synchronize()
    return out, sl


@pytest.mark.parametrize("shape", [
    dict(G=2, D=128, P=32, chunk=(300, 200, 600)),
    dict(G=7, D=128, P=16, chunk=(0, 130, 150)),
    dict(G=1, D=64, P=64, chunk=(37, 64, 200)),
    dict(G=8, D=128, P=128, chunk=(64, 257, 321)),
    dict(G=4, D=64, P=256, chunk=(9000, 200, 9300)),   # key ranges split and merged
    dict(G=2, D=128, P=16, chunk=(9000, 200, 9300)),
], ids=lambda d: f"G{d['G']}-D{d['D']}-P{d['P']}-at{d['chunk'][0]}")
def test_tiles_only_launch_bits_equal_mixed_launch(shape):
    """A call whose rows are all in a tile-path chunk runs the tile CTAs in a
    launch of their own shape; the chunk rows' bits must equal those the same
    rows get beside decode rows, and match the oracle."""
    G, D, P = shape["G"], shape["D"], shape["P"]
    wl = W.chunked_step(80 + G + D + P, [shape["chunk"]], decode_ctx=[30, 700], Hq=2 * G, Hkv=2, D=D, P=P)
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    mixed = st.out.view(torch.int16).clone()
    out, sl = chunk_alone(st, wl)
    assert int(st.status.item()) == 0
    assert torch.equal(out.view(torch.int16), mixed[sl]), "chunk rows differ between the two launches"
    kp, vp = oracle_pools(wl)
    ref = oracle_out(wl, kp, vp)[sl]
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(out)).astype(np.float64)
    assert_close(got, ref, wl, "chunk alone")


def test_tiles_only_launch_step_and_timeout():
    """pa_step on a call of chunk rows only (the append, then the tile launch
    as its dependent) equals the two calls; an injected stall in the tile
    launch reports PA_ERR_TIMEOUT and the next call is exact again."""
    wl = W.chunked_step(91, [(500, 256, 800)])
    a = pa_setup.upload(wl)
    a.append_step()
    a.attend()
    b = pa_setup.upload(wl)
    b.step()
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))  # NaN-poisoned slots: compare bits
    assert torch.equal(a.v_pool.view(torch.int16), b.v_pool.view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    good = a.out.view(torch.int16).clone()
    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        a.status.zero_()
        a.attend()
        torch.cuda.synchronize()
        code = int(a.status.item())
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert code == pa.PA_ERR_TIMEOUT
    a.status.zero_()
    a.attend()
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0
    assert torch.equal(a.out.view(torch.int16), good)


def test_long_prefill_sampled_rows():
    """The prefill-step workload of the benchmark (one 4096-token causal chunk,
    512 tiles, no decode rows): pool bytes equal the oracle's; rows sampled
    across the chunk (tile edges, the first and last rows) match the oracle."""
    wl = W.long_prefill()
    st = pa_setup.upload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    assert pa_setup.to_numpy(st.k_pool).tobytes() == kp.tobytes()
    assert pa_setup.to_numpy(st.v_pool).tobytes() == vp.tobytes()
    rows = np.array([0, 1, 63, 64, 65, 127, 128, 1000, 2047, 2048, 3071, 4031, 4032, 4094, 4095])
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)[rows]).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp, rows=rows), wl, "long prefill, sampled rows")
