"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

  * pool bytes after append equal the oracle's, byte for byte (untouched
    NaN-poisoned slots included);
  * attention outputs within the tolerance: |gpu - ref| <= 2e-3 or <= 1e-2 |ref|
    for bf16/fp8 K/V, 1e-5 / 1e-5 for f32 K/V;
  * every shape at a size the oracle finishes in seconds (several pages per
    sequence, split boundaries, partial last pages), and the full sizes on all
    rows or on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


def run_step(wl):
    st = pa_setup.upload(wl)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    return st


def check_pools(st, kp, vp, pages=None):
    gk, gv = pa_setup.to_numpy(st.k_pool), pa_setup.to_numpy(st.v_pool)
    if pages is None:
        assert gk.tobytes() == kp.tobytes(), "K pool differs from the oracle's"
        assert gv.tobytes() == vp.tobytes(), "V pool differs from the oracle's"
    else:
        pages = np.asarray(sorted(pages))
        assert gk[pages].tobytes() == kp[pages].tobytes(), "K pages differ from the oracle's"
        assert gv[pages].tobytes() == vp[pages].tobytes(), "V pages differ from the oracle's"


@pytest.mark.parametrize("name", list(W.SMALL))
def test_small_configs_match_oracle(name):
    wl = W.SMALL[name]()
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    ref = oracle_out(wl, kp, vp)
    got = pa_setup.to_numpy(st.out)
    got = got.astype(np.float64) if wl.q_dtype == W.F32 else W.bf16_bits_to_f32(got).astype(np.float64)
    assert_close(got, ref, wl, name)


@pytest.mark.parametrize("split", [64, 256, 2048])
def test_split_sizes_match_oracle(split):
    old = pa.get_split_tokens()
    pa.set_split_tokens(split)
    try:
        wl = W.batched_decode(n_seqs=12, ctx_hi=1500)
        st = run_step(wl)
        assert int(st.status.item()) == 0
        kp, vp = oracle_pools(wl)
        got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
        assert_close(got, oracle_out(wl, kp, vp), wl, f"split {split}")
    finally:
        pa.set_split_tokens(old)


@pytest.mark.parametrize("P", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("kv_dtype", [W.F32, W.BF16, W.E4M3])
def test_page_sizes_and_dtypes(P, kv_dtype):
    q_dtype = W.F32 if kv_dtype == W.F32 else W.BF16
    rng = np.random.default_rng(P * 10 + kv_dtype)
    ctx = rng.integers(1, 700, size=9).tolist() + [1, P, P + 1]
    wl = W._decode_workload("pt", 77 + P + kv_dtype, ctx, 8, 2, 128 if P != 64 else 64, P, kv_dtype, q_dtype,
                            max_ctx=704, spare_pages=5, description="page/dtype sweep")
    if kv_dtype == W.E4M3:
        wl.k_scale, wl.v_scale = 0.0123, 0.0101
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    got = pa_setup.to_numpy(st.out)
    got = got.astype(np.float64) if q_dtype == W.F32 else W.bf16_bits_to_f32(got).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, f"P{P} kv{kv_dtype}")


@pytest.mark.parametrize("P", [16, 64, 128, 256])
@pytest.mark.parametrize("G", [3, 7])
def test_bf16_tensor_core_units_page_sizes(G, P):
    """The bf16 tensor-core decode units (D 128, G 3..8): 32-token stages that are
    two pages, one page or part of a page, contexts ending on and just past
    stage and page boundaries."""
    ctx = [1, 31, 32, 33, P - 1, P, P + 1, 2 * P + 5, 700]
    wl = W._decode_workload("bfmma", 1300 + 11 * G + P, ctx, 2 * G, 2, 128, P, W.BF16, W.BF16, max_ctx=768,
                            spare_pages=4, description="bf16 tensor-core units, page sizes")
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, f"bf16 mma G{G} P{P}")


@pytest.mark.parametrize("G", [1, 3, 5, 6, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_group_sizes(G, D):
    wl = W._decode_workload("gs", 900 + G * 7 + D, [3, 77, 300, 1111], 2 * G, 2, D, 32, W.BF16, W.BF16,
                            max_ctx=1200, spare_pages=2, description="group sweep")
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, f"G{G} D{D}")


def test_single_position_returns_value_exactly():
    wl = W._decode_workload("one", 5, [1] * 16, 8, 2, 128, 32, W.BF16, W.BF16, max_ctx=32, spare_pages=0,
                            description="single position")
    st = run_step(wl)
    got = pa_setup.to_numpy(st.out)  # bf16 bits
    for r in range(wl.n_rows):
        for g in range(wl.Hq):
            assert got[r, g].tobytes() == wl.v_new[r, g // 4].tobytes()


def test_identical_keys_give_mean_of_values():
    wl = W.batched_decode(n_seqs=8, ctx_hi=900)
    st = pa_setup.upload(wl)
    st.k_pool.fill_(0.5)  # every key identical: uniform weights
    st.k_new.fill_(0.5)
    st.append_step()
    st.attend()
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    vf = W.bf16_bits_to_f32(wl.hist_v).astype(np.float64)
    vn = W.bf16_bits_to_f32(wl.v_new).astype(np.float64)
    G = wl.Hq // wl.Hkv
    for r in range(wl.n_rows):
        rows = vf[wl.hist_seq == r]
        allv = np.concatenate([rows, vn[r:r + 1]])
        mean = allv.mean(axis=0)  # [Hkv, D]
        assert_close(got[r], np.repeat(mean, G, axis=0), wl, "mean of V")


def test_fp8_encoder_matches_oracle_on_float_sweep():
    """The GPU e4m3 conversion (through append with scale 1, f32 rows in) against
    the oracle's encoder on every upper-16-bit pattern with a spread of low bits."""
    hi = (np.arange(1 << 16, dtype=np.uint32) << 16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000], np.uint32)
    x = (hi[:, None] | lows[None, :]).reshape(-1).view(np.float32)
    x = x[~np.isnan(x)]
    n = (x.size // 128) * 128
    x = x[:n].reshape(-1, 1, 128)
    rows = x.shape[0]
    bt = torch.arange(rows, dtype=torch.int32, device="cuda").reshape(1, rows)
    kp = torch.zeros((rows, 1, 16, 128), dtype=torch.uint8, device="cuda")
    vp = torch.zeros_like(kp)
    pool = pa.Pool(kp, vp, 1.0, 1.0)
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.arange(rows, dtype=torch.int32, device="cuda") * 16
    pa.append_kv(pool, xt, xt, torch.zeros(rows, dtype=torch.int32, device="cuda"), pos, bt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = kp[:, 0, 0, :].cpu().numpy().reshape(-1)
    ref = oracle.e4m3_from_f32_array(x.reshape(-1))
    np.testing.assert_array_equal(got, ref)


def _oracle_codes(bits_lo: int, n: int, threads: int) -> np.ndarray:
    """The oracle's e4m3 codes of the binary32 patterns bits_lo .. bits_lo + n - 1,
    encoded in pieces on the host cores."""
    import concurrent.futures as cf
    x = np.arange(bits_lo, bits_lo + n, dtype=np.uint32).view(np.float32)
    out = np.empty(n, dtype=np.uint8)
    piece = (n + threads - 1) // threads

    def enc(i):
        a, b = i * piece, min(n, (i + 1) * piece)
        if a < b:
            out[a:b] = oracle.e4m3_from_f32_array(x[a:b])

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(enc, range(threads)))
    return out


def test_fp8_append_encoder_on_every_binary32_pattern():
    """pa_append_kv into an e4m3 pool with scale 1 (x / 1 = x) on all 2^32
    binary32 patterns -- NaNs, infinities, subnormals and both zeros
    included -- against the oracle's encoder, code for code.  2^26 patterns
    per call as the K rows and the next 2^26 as the V rows; one sequence of
    8192 positions, 64 kv heads x 128 elements, 256-token pages."""
    n, Hkv, D, P = 1 << 26, 64, 128, 256
    rows = n // (Hkv * D)
    pages = rows // P
    kp = torch.zeros((pages, Hkv, P, D), dtype=torch.uint8, device="cuda")
    vp = torch.zeros_like(kp)
    pool = pa.Pool(kp, vp, 1.0, 1.0)
    bt = torch.arange(pages, dtype=torch.int32, device="cuda").reshape(1, pages)
    seq = torch.zeros(rows, dtype=torch.int32, device="cuda")
    pos = torch.arange(rows, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    threads = oracle.host_cores()

    def patterns(lo):
        b = torch.arange(lo, lo + n, dtype=torch.int64, device="cuda")
        b = torch.where(b >= 1 << 31, b - (1 << 32), b).to(torch.int32)
        return b.view(torch.float32).reshape(rows, Hkv, D)

    for lo in range(0, 1 << 32, 2 * n):
        pa.append_kv(pool, patterns(lo), patterns(lo + n), seq, pos, bt, status=status)
        # [page][head][slot][d] -> [row = page * P + slot][head][d]: the input order
        got_k = kp.permute(0, 2, 1, 3).reshape(-1).cpu().numpy()
        got_v = vp.permute(0, 2, 1, 3).reshape(-1).cpu().numpy()
        assert int(status.item()) == 0
        for got, base in ((got_k, lo), (got_v, lo + n)):
            ref = _oracle_codes(base, n, threads)
            if not np.array_equal(got, ref):
                i = int(np.flatnonzero(got != ref)[0])
                raise AssertionError(f"pattern {base + i:#010x}: GPU code {got[i]:#04x}, oracle {ref[i]:#04x} "
                                     f"({int(np.count_nonzero(got != ref))} of {n} differ in this piece)")


# ------------------------------------------------------------ full sizes ----

def _sampled(wl, rows, what):
    st = run_step(wl)
    assert int(st.status.item()) == 0
    seqs = sorted(set(int(s) for s in wl.seq_ids[rows]))
    kp, vp = oracle_pools(wl, rows_of_seqs=seqs)
    pages = set(int(p) for p in wl.block_tables[seqs].reshape(-1) if p >= 0)
    check_pools(st, kp, vp, pages)
    ref = oracle_out(wl, kp, vp, rows=rows)
    got = pa_setup.to_numpy(st.out)[rows]
    got = got.astype(np.float64) if wl.q_dtype == W.F32 else W.bf16_bits_to_f32(got).astype(np.float64)
    return assert_close(got, ref, wl, what)


def test_full_batched_decode_all_rows():
    wl = W.batched_decode()
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, "batched decode, 512 rows")


def test_full_shared_prefix_all_rows():
    wl = W.shared_prefix()
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, "shared prefix, 768 rows")


def test_full_mixed_step_all_rows():
    wl = W.mixed_step()
    st = run_step(wl)
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    check_pools(st, kp, vp)
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, "mixed step, 512 rows")


def test_full_long_context_sampled_rows():
    wl = W.long_context()
    _sampled(wl, np.array([0, 17, 40, 63]), "long context, 4 of 64 rows")


def test_full_batched_decode_fp8_sampled_rows():
    wl = W.batched_decode_fp8()
    _sampled(wl, np.array([0, 1, 100, 255, 300, 511]), "batched decode fp8, 6 of 512 rows")


def test_full_long_context_fp8_sampled_rows():
    wl = W.long_context_fp8()
    _sampled(wl, np.array([0, 33, 63]), "long context fp8, 3 of 64 rows")
