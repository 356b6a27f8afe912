"""GPU parity of the tensor-core decode units (e4m3 K/V, head_dim 128, bf16
queries, 1..8 query heads per kv head) against the CPU oracle, and the same
failure reporting and bit-identity guarantees as the SIMT units.

The shapes span: every group size, every page size (one, two or several
tensor-map boxes per 32-token stage), contexts that end on and just past
stage and page boundaries, split-KV rows, queries whose largest element is far
above or below the f16 range (the power-of-two query scaling), and f32
queries (which take the SIMT units)."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu

CTX = [1, 2, 31, 32, 33, 64, 65, 129, 300, 777]


def fp8_workload(seed, G, P, ctx=CTX, q_dtype=W.BF16, max_ctx=800, Hkv=2):
    wl = W._decode_workload("fp8mma", seed, ctx, G * Hkv, Hkv, 128, P, W.E4M3, q_dtype, max_ctx=max_ctx,
                            spare_pages=3, description="e4m3 tensor-core decode")
    wl.k_scale, wl.v_scale = 0.0173, 0.0119
    return wl


def check(wl, what):
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    got = pa_setup.to_numpy(st.out)
    got = got.astype(np.float64) if wl.q_dtype == W.F32 else W.bf16_bits_to_f32(got).astype(np.float64)
    return st, assert_close(got, oracle_out(wl, kp, vp), wl, what)


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_groups_and_pages(G, P):
    check(fp8_workload(500 + 10 * G + P, G, P), f"G{G} P{P}")


def test_f32_queries():
    check(fp8_workload(71, 7, 32, q_dtype=W.F32), "f32 q")


@pytest.mark.parametrize("log2_scale", [-40, -12, 12, 40])
def test_query_magnitudes(log2_scale):
    """Queries scaled by 2^k (exact in bf16): the kernel's power-of-two query
    scaling must keep them representable in f16 whatever their size."""
    wl = fp8_workload(90 + log2_scale, 7, 32)
    qf = W.bf16_bits_to_f32(wl.q) * np.float32(2.0 ** log2_scale)
    wl.q = W.to_bf16_bits(qf)
    wl.softmax_scale = float(2.0 ** (-log2_scale)) / np.sqrt(128.0)  # keep the scores' spread
    check(wl, f"q * 2^{log2_scale}")


@pytest.mark.parametrize("split", [64, 256, 1024])
def test_split_rows(split):
    old = pa.get_split_tokens()
    pa.set_split_tokens(split)
    try:
        check(fp8_workload(33 + split, 7, 32, ctx=[5, 300, 1500, 2047, 2048, 2049], max_ctx=2112), f"split {split}")
    finally:
        pa.set_split_tokens(old)


def test_shared_prefix_batch_composition_bit_identical():
    wl = W.shared_prefix(n_seqs=40)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()

    def rows_out(rows):
        rows = torch.as_tensor(np.asarray(rows), dtype=torch.long, device="cuda")
        q = st.q[rows].contiguous()
        out = torch.empty_like(q)
        wsb = pa.workspace_bytes(st.pool, q.shape[0], wl.Hq, wl.max_blocks)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda") if wsb else None
        pa.attention(st.pool, q, st.seq_ids[rows].contiguous(), st.positions[rows].contiguous(), st.block_tables,
                     out, softmax_scale=wl.softmax_scale, workspace=ws, status=st.status)
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        return out.view(torch.int16).cpu().numpy()

    n = wl.n_rows
    full = rows_out(np.arange(n))
    for r in (0, 7, n - 1):
        assert rows_out([r]).tobytes() == full[r:r + 1].tobytes(), f"row {r} alone differs"
    perm = np.random.default_rng(5).permutation(n)
    assert rows_out(perm).tobytes() == full[perm].tobytes(), "shuffled batch differs"
    for _ in range(5):
        assert rows_out(np.arange(n)).tobytes() == full.tobytes(), "repeat differs"


def test_bad_page_and_stall_reported():
    wl = fp8_workload(12, 4, 32)
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    good = st.out.clone()

    bt = st.block_tables.clone()
    bt[8, 0] = wl.num_pages + 1  # row 8 (context 300) reads a page id past the pool
    out = torch.empty_like(st.q)
    st.status.zero_()
    pa.attention(st.pool, st.q, st.seq_ids, st.positions, bt, out, softmax_scale=wl.softmax_scale,
                 workspace=st.workspace, status=st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == pa.PA_ERR_OUT_OF_RANGE
    assert torch.count_nonzero(out[8].float()) == 0
    keep = [i for i in range(wl.n_rows) if i != 8]
    assert torch.equal(out[keep].view(torch.int16), good[keep].view(torch.int16))

    pa.set_wait_limit(1000)
    pa.debug_stall_waits(True)
    try:
        st.status.zero_()
        pa.attention(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, out,
                     softmax_scale=wl.softmax_scale, workspace=st.workspace, status=st.status)
        torch.cuda.synchronize()
    finally:
        pa.debug_stall_waits(False)
        pa.set_wait_limit(0)
    assert int(st.status.item()) == pa.PA_ERR_TIMEOUT
    st.status.zero_()
    pa.attention(st.pool, st.q, st.seq_ids, st.positions, st.block_tables, out,
                 softmax_scale=wl.softmax_scale, workspace=st.workspace, status=st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    assert torch.equal(out.view(torch.int16), good.view(torch.int16))


def value_scaled(wl, k, per_head=False):
    """K and V multiplied by 2^k (exact in bf16) with the fp8 scales calibrated
    on the scaled values (amax / 448, per tensor or per kv head) and the
    softmax scale divided by 2^k: the stored codes and the scores do not
    change, every output grows by 2^k, and so does any error the P.V product
    makes relative to the values."""
    f = np.float32(2.0 ** k)
    for name in ("hist_k", "hist_v", "k_new", "v_new"):
        setattr(wl, name, W._cast(W.as_f32(getattr(wl, name), wl.in_dtype) * f, wl.in_dtype))
    wl.softmax_scale = float(2.0 ** (-k)) / np.sqrt(128.0)
    if not per_head:
        return W._with_fp8_scales(wl)
    ax = (0, 2)
    amax_k = np.maximum(np.abs(W.as_f32(wl.hist_k, wl.in_dtype)).max(axis=ax),
                        np.abs(W.as_f32(wl.k_new, wl.in_dtype)).max(axis=ax))
    amax_v = np.maximum(np.abs(W.as_f32(wl.hist_v, wl.in_dtype)).max(axis=ax),
                        np.abs(W.as_f32(wl.v_new, wl.in_dtype)).max(axis=ax))
    wl.k_scale = (amax_k.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    wl.v_scale = (amax_v.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    return wl


@pytest.mark.parametrize("k", [3, 6, 7])
@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_values_far_from_unit_scale(G, P, k):
    """The P.V product must see each softmax weight to far better than f16's
    2^-11: its error grows with the values' magnitude, and at 2^6..2^7 an
    output that cancels to near zero would miss the absolute tolerance."""
    wl = value_scaled(fp8_workload(700 + 10 * G + P + k, G, P), k)
    check(wl, f"G{G} P{P} values x 2^{k}")


@pytest.mark.parametrize("G", [1, 4, 7, 8])
def test_values_far_from_unit_scale_per_head_scales(G):
    """The same with one fp8 scale per kv head (4 kv heads, each calibrated on
    its own values), values x 2^7."""
    wl = value_scaled(fp8_workload(800 + G, G, 32, Hkv=4), 7, per_head=True)
    check(wl, f"G{G} per-head scales, values x 2^7")
