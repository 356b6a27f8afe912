"""Bit-identity of a row's output across batch compositions ("GPU inference
engine engineering", section "The same bits in any batch": alone or in a
batch, shuffled, under repeated runs), and across physical page placement."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def attend_rows(st, rows, chunks=()):
    """Attention of a subset of the step's rows (after the step's append), as bf16 bits."""
    rows = torch.as_tensor(np.asarray(rows), dtype=torch.long, device="cuda")
    q = st.q[rows].contiguous()
    out = torch.empty_like(q)
    n = q.shape[0]
    wsb = pa.workspace_bytes(st.pool, n, st.wl.Hq, st.wl.max_blocks, chunks)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    pa.attention(st.pool, q, st.seq_ids[rows].contiguous(), st.positions[rows].contiguous(), st.block_tables, out,
                 chunks=chunks, workspace=ws, status=st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return out.view(torch.int16).cpu().numpy()


@pytest.fixture(scope="module")
def step():
    wl = W.batched_decode(n_seqs=64)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    return st


def test_alone_vs_batch_vs_shuffled_vs_repeats(step):
    n = step.wl.n_rows
    full = attend_rows(step, np.arange(n))
    for r in (0, 5, 33, n - 1):
        assert attend_rows(step, [r]).tobytes() == full[r:r + 1].tobytes(), f"row {r} alone differs"
    rng = np.random.default_rng(3)
    for _ in range(3):
        perm = rng.permutation(n)
        shuf = attend_rows(step, perm)
        assert shuf.tobytes() == full[perm].tobytes(), "shuffled batch differs"
    sub = rng.choice(n, size=7, replace=False)
    assert attend_rows(step, sub).tobytes() == full[sub].tobytes()
    for _ in range(10):
        assert attend_rows(step, np.arange(n)).tobytes() == full.tobytes(), "repeat differs"


def test_duplicated_rows_in_one_batch(step):
    full = attend_rows(step, np.arange(step.wl.n_rows))
    rows = [3, 3, 9, 3]
    got = attend_rows(step, rows)
    assert got.tobytes() == full[rows].tobytes()


def test_page_permutation_bit_identical(step):
    wl = step.wl
    full = attend_rows(step, np.arange(wl.n_rows))
    perm = torch.randperm(wl.num_pages, generator=torch.Generator().manual_seed(9)).cuda()
    k2 = torch.empty_like(step.k_pool)
    v2 = torch.empty_like(step.v_pool)
    k2[perm] = step.k_pool
    v2[perm] = step.v_pool
    bt = step.block_tables.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32).contiguous()
    pool2 = pa.Pool(k2, v2)
    out = torch.empty_like(step.q)
    wsb = pa.workspace_bytes(pool2, wl.n_rows, wl.Hq, wl.max_blocks)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    pa.attention(pool2, step.q, step.seq_ids, step.positions, bt2, out, workspace=ws, status=step.status)
    torch.cuda.synchronize()
    assert out.view(torch.int16).cpu().numpy().tobytes() == full.tobytes()


def test_decode_rows_unchanged_beside_a_prefill_chunk():
    wl = W.mixed_step(n_decode=48, ctx_hi=1024)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    dec = wl.decode_rows()
    together = attend_rows(st, np.arange(wl.n_rows), chunks=wl.chunks)
    alone = attend_rows(st, dec)
    assert together[dec].tobytes() == alone.tobytes()


@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (28, 4), (32, 4)])
def test_decode_rows_unchanged_beside_a_chunk_on_tensor_core_units(Hq, Hkv):
    """G >= 3 (bf16, D 128): decode rows run on the tensor-core units, inside
    the mixed launch as in a decode-only launch; their bits must not change."""
    wl = W.chunked_step(71 + Hq, chunks=[(200, 180, 416)], decode_ctx=[5, 64, 333, 700, 1029], Hq=Hq, Hkv=Hkv)
    st = pa_setup.upload(wl)
    st.append_step()
    torch.cuda.synchronize()
    dec = wl.decode_rows()
    together = attend_rows(st, np.arange(wl.n_rows), chunks=wl.chunks)
    alone = attend_rows(st, dec)
    assert together[dec].tobytes() == alone.tobytes()
    shuffled = np.random.default_rng(1).permutation(dec)
    assert attend_rows(st, shuffled).tobytes() == together[shuffled].tobytes()
