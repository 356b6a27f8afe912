"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * brute force: contiguous, un-paged attention written with numpy matrix
    products and scipy's softmax on the same stored values;
  * invariants: random permutation of the physical pages (bit-identical);
  * closed forms: identical keys or q = 0 give the mean of V; a single
    position returns its V exactly;
  * library routines for the two encoders: torch's fp32->bf16 cast (RNE) and
    torch's float8_e4m3fn cast inside the non-saturating range;
  * the OCP E4M3 definition, code by code, and the page-count figures the
    pages print.
A separate test (test_oracle_mutants.py) plants plausible mistakes in a copy
of the oracle and checks that these pins catch each one.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import workloads as W

RNG = np.random.default_rng(12345)


# --------------------------------------------------------------- helpers ----

def make_case(rng, L_list, Hq, Hkv, D, P, kv_dtype=W.F32, in_dtype=W.F32, q_dtype=W.F32,
              num_pages=None, scale=(1.0, 1.0), shuffle=True):
    """A small paged case built with the oracle's own append: sequences with
    contexts L_list, one decode row each at position L-1."""
    pages = [(L + P - 1) // P for L in L_list]
    max_blocks = max(pages)
    if num_pages is None:
        num_pages = sum(pages) + 3
    perm = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    bt = np.full((len(L_list), max_blocks), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[k:k + n]
        k += n
    seq = np.repeat(np.arange(len(L_list), dtype=np.int32), L_list)
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in L_list])
    x_k = rng.standard_normal((len(seq), Hkv, D)).astype(np.float32)
    x_v = rng.standard_normal((len(seq), Hkv, D)).astype(np.float32)
    if in_dtype == W.BF16:
        x_k, x_v = W.to_bf16_bits(x_k), W.to_bf16_bits(x_v)
    wl = W.Workload(name="pin", Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=kv_dtype, in_dtype=in_dtype,
                    q_dtype=q_dtype, num_pages=num_pages, block_tables=bt, hist_seq=seq, hist_pos=pos,
                    hist_k=x_k, hist_v=x_v, seq_ids=np.arange(len(L_list), dtype=np.int32),
                    positions=np.array(L_list, dtype=np.int32) - 1, q=None, k_new=None, v_new=None,
                    k_scale=scale[0], v_scale=scale[1])
    kp, vp = wl.empty_pool(), wl.empty_pool()
    st = oracle.append(x_k, x_v, in_dtype, seq, pos, bt, num_pages, P, Hkv, D, kv_dtype, scale[0],
                       scale[1], kp, vp)
    assert st == 0
    q = rng.standard_normal((len(L_list), Hq, D)).astype(np.float32)
    if q_dtype == W.BF16:
        q = W.to_bf16_bits(q)
    wl.q = q
    return wl, kp, vp, x_k, x_v, seq, pos


def stored_values(x, in_dtype, kv_dtype, scale):
    """The values the pool holds for input rows x, as float64 (fp8: code value x scale)."""
    xf = W.as_f32(x, in_dtype)
    if kv_dtype == W.F32:
        return xf.astype(np.float64)
    if kv_dtype == W.BF16:
        return W.bf16_bits_to_f32(W.to_bf16_bits(xf)).astype(np.float64)
    codes = oracle.e4m3_from_f32_array((xf / np.float32(scale)).astype(np.float32))
    table = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    return table[codes] * float(np.float32(scale))  # the scale travels as binary32


def brute_force(wl, x_k, x_v, seq, pos, softmax_scale=None):
    """Un-paged attention: gather each sequence's keys by position from the input
    rows, then softmax(scale * q K^T) V with numpy / scipy in float64."""
    kv = stored_values(x_k, wl.in_dtype, wl.kv_dtype, wl.k_scale)
    vv = stored_values(x_v, wl.in_dtype, wl.kv_dtype, wl.v_scale)
    G = wl.Hq // wl.Hkv
    sc = 1.0 / math.sqrt(wl.D) if softmax_scale is None else softmax_scale
    qf = W.as_f32(wl.q, wl.q_dtype).astype(np.float64)
    out = np.zeros((wl.n_rows, wl.Hq, wl.D))
    for r in range(wl.n_rows):
        s, p = wl.seq_ids[r], wl.positions[r]
        idx = np.nonzero(seq == s)[0]
        idx = idx[np.argsort(pos[idx])][: p + 1]
        assert np.array_equal(pos[idx], np.arange(p + 1))
        for g in range(wl.Hq):
            Kc = kv[idx, g // G, :]
            Vc = vv[idx, g // G, :]
            w = softmax(sc * (Kc @ qf[r, g]))
            out[r, g] = w @ Vc
    return out


def run_oracle(wl, kp, vp, softmax_scale=0.0, n_threads=1):
    return oracle.attention(wl.q, wl.q_dtype, wl.Hq, wl.seq_ids, wl.positions, wl.block_tables,
                            wl.num_pages, wl.P, wl.Hkv, wl.D, wl.kv_dtype, wl.k_scale, wl.v_scale,
                            kp, vp, softmax_scale=softmax_scale, n_threads=n_threads)


# ------------------------------------------------------ p1: brute force ----

@pytest.mark.parametrize("D", [4, 64])
@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("P", [1, 4, 32])
def test_matches_contiguous_brute_force_f32(D, G, P):
    rng = np.random.default_rng(1000 * D + 10 * G + P)
    L_list = [int(x) for x in rng.integers(1, 71, size=3)] + [1]
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, L_list, Hq=2 * G, Hkv=2, D=D, P=P)
    got = run_oracle(wl, kp, vp)
    ref = brute_force(wl, xk, xv, seq, pos)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kv_dtype,in_dtype", [(W.BF16, W.BF16), (W.BF16, W.F32), (W.E4M3, W.BF16),
                                               (W.E4M3, W.F32), (W.F32, W.BF16)])
def test_matches_brute_force_storage_dtypes(kv_dtype, in_dtype):
    rng = np.random.default_rng(7 + kv_dtype * 10 + in_dtype)
    L_list = [3, 40, 65]
    scale = (0.0123, 0.0311) if kv_dtype == W.E4M3 else (1.0, 1.0)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, L_list, Hq=8, Hkv=2, D=64, P=32, kv_dtype=kv_dtype,
                                             in_dtype=in_dtype, q_dtype=W.BF16, scale=scale)
    got = run_oracle(wl, kp, vp)
    ref = brute_force(wl, xk, xv, seq, pos)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_softmax_scale_argument():
    rng = np.random.default_rng(99)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [17, 50], Hq=4, Hkv=2, D=16, P=4)
    for sc in (0.05, 0.7, 2.5):
        np.testing.assert_allclose(run_oracle(wl, kp, vp, softmax_scale=sc),
                                   brute_force(wl, xk, xv, seq, pos, softmax_scale=sc), rtol=1e-12, atol=1e-13)
    # scale <= 0 means 1/sqrt(D)
    np.testing.assert_array_equal(run_oracle(wl, kp, vp, 0.0), run_oracle(wl, kp, vp, -1.0))
    np.testing.assert_allclose(run_oracle(wl, kp, vp, 0.0), run_oracle(wl, kp, vp, 0.25), rtol=1e-15)


# --------------------------------------------- p2: page permutation ----

def test_page_permutation_is_bit_identical():
    rng = np.random.default_rng(5)
    L_list = [5, 33, 64, 100]
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, L_list, Hq=8, Hkv=2, D=64, P=32, num_pages=16)
    base = run_oracle(wl, kp, vp)
    for trial in range(3):
        perm = rng.permutation(wl.num_pages)  # physical page i moves to perm[i]
        kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
        kp2[perm], vp2[perm] = kp, vp
        bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
        wl2 = W.Workload(**{**wl.__dict__, "block_tables": bt2})
        out = run_oracle(wl2, kp2, vp2)
        assert out.tobytes() == base.tobytes()


def test_threads_do_not_change_bits():
    rng = np.random.default_rng(6)
    wl, kp, vp, *_ = make_case(rng, [9, 31, 77, 120, 5, 64], Hq=8, Hkv=2, D=32, P=16)
    a = run_oracle(wl, kp, vp, n_threads=1)
    b = run_oracle(wl, kp, vp, n_threads=4)
    assert a.tobytes() == b.tobytes()


def test_unused_poisoned_slots_never_read():
    """The pool starts NaN-poisoned; slots past a row's position and pages no
    table points to must not reach the output."""
    rng = np.random.default_rng(8)
    wl, kp, vp, *_ = make_case(rng, [5, 33, 64, 100], Hq=8, Hkv=2, D=64, P=32, num_pages=16)
    assert np.isnan(kp).any()
    assert np.isfinite(run_oracle(wl, kp, vp)).all()


# ------------------------------------------------------ p3/p4: closed forms ----

def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(11)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [1, 7, 45], Hq=4, Hkv=1, D=8, P=4)
    kp[...] = 0.37  # every key the same vector
    out = run_oracle(wl, kp, vp)
    for r in range(wl.n_rows):
        s, p = wl.seq_ids[r], wl.positions[r]
        idx = np.nonzero(seq == s)[0][: p + 1]
        mean_v = xv[idx, 0, :].astype(np.float64).mean(axis=0)
        for g in range(wl.Hq):
            np.testing.assert_allclose(out[r, g], mean_v, rtol=1e-13, atol=1e-14)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(12)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [3, 30], Hq=2, Hkv=2, D=8, P=8)
    wl.q[...] = 0.0
    out = run_oracle(wl, kp, vp)
    for r in range(wl.n_rows):
        idx = np.nonzero(seq == wl.seq_ids[r])[0]
        for g in range(2):
            np.testing.assert_allclose(out[r, g], xv[idx, g, :].astype(np.float64).mean(axis=0), rtol=1e-13)


@pytest.mark.parametrize("kv_dtype", [W.F32, W.BF16, W.E4M3])
def test_single_position_returns_its_value_exactly(kv_dtype):
    rng = np.random.default_rng(13 + kv_dtype)
    in_dtype = W.F32
    scale = (0.02, 0.03) if kv_dtype == W.E4M3 else (1.0, 1.0)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [1, 1, 1], Hq=6, Hkv=3, D=16, P=8, kv_dtype=kv_dtype,
                                             in_dtype=in_dtype, scale=scale)
    out = run_oracle(wl, kp, vp)
    stored = stored_values(xv, in_dtype, kv_dtype, scale[1])
    for r in range(3):
        for g in range(6):
            assert np.array_equal(out[r, g], stored[r, g // 2])


def test_hand_worked_two_token_case():
    """q = [ln 3 * 2, 0], keys [0,0] and [1,0], scale 1/sqrt(D) with D = 4 gives
    scores 0 and ln 3, weights 1/4 and 3/4: out = v0/4 + 3 v1/4."""
    D = 4
    k = np.zeros((2, 1, D), np.float32)
    k[1, 0, 0] = 1.0
    v = np.array([[[4.0, 0.0, -8.0, 1.0]], [[0.0, 4.0, 8.0, 1.0]]], np.float32)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = np.float32(2.0 * math.log(3.0))  # times 1/sqrt(4) = ln 3
    bt = np.array([[0]], np.int32)
    kp = np.zeros((1, 1, 2, D), np.float32)
    vp = np.zeros_like(kp)
    assert oracle.append(k, v, W.F32, np.zeros(2, np.int32), np.arange(2, dtype=np.int32), bt, 1, 2, 1, D,
                         W.F32, 1.0, 1.0, kp, vp) == 0
    out = oracle.attention(q, W.F32, 1, np.zeros(1, np.int32), np.array([1], np.int32), bt, 1, 2, 1, D,
                           W.F32, 1.0, 1.0, kp, vp)
    s1 = float(np.float32(2.0 * math.log(3.0))) * 0.5  # the float32 query, exactly as stored
    w1 = math.exp(s1) / (1.0 + math.exp(s1))
    expect = (1 - w1) * v[0, 0].astype(np.float64) + w1 * v[1, 0].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14)
    np.testing.assert_allclose(out[0, 0], [1.0, 3.0, 4.0, 1.0], rtol=1e-6)


# ----------------------------------------------------------- p5: GQA ----

def test_gqa_group_one_is_mha_and_shared_query_heads_agree():
    rng = np.random.default_rng(21)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [12, 40], Hq=4, Hkv=4, D=16, P=8)
    np.testing.assert_allclose(run_oracle(wl, kp, vp), brute_force(wl, xk, xv, seq, pos), rtol=1e-12)
    wl2, kp2, vp2, *_ = make_case(np.random.default_rng(22), [12, 40], Hq=8, Hkv=2, D=16, P=8)
    wl2.q[:, 1] = wl2.q[:, 0]  # heads 0 and 1 share kv head 0
    wl2.q[:, 5] = wl2.q[:, 4]  # heads 4 and 5 share kv head 1
    out = run_oracle(wl2, kp2, vp2)
    assert np.array_equal(out[:, 0], out[:, 1]) and np.array_equal(out[:, 4], out[:, 5])
    assert not np.array_equal(out[:, 0], out[:, 4])


# ------------------------------------------------------------ p6: append ----

def test_append_roundtrip_and_page_boundary():
    rng = np.random.default_rng(31)
    P, H, D = 4, 2, 8
    bt = np.array([[3, 0, 5], [1, 4, 2]], np.int32)
    pos = np.array([3, 4, 0, 7, 8], np.int32)  # slot P-1 then slot 0 of the next page, etc.
    seq = np.array([0, 0, 1, 1, 1], np.int32)
    for kv_dtype, in_dtype in [(W.F32, W.F32), (W.BF16, W.BF16), (W.F32, W.BF16)]:
        x = rng.standard_normal((5, H, D)).astype(np.float32)
        if in_dtype == W.BF16:
            x = W.to_bf16_bits(x)
        np_t = np.float32 if kv_dtype == W.F32 else np.uint16
        kp = np.zeros((6, H, P, D), np_t)
        vp = np.zeros_like(kp)
        assert oracle.append(x, x, in_dtype, seq, pos, bt, 6, P, H, D, kv_dtype, 1, 1, kp, vp) == 0
        for r in range(5):
            page = bt[seq[r], pos[r] // P]
            got = kp[page, :, pos[r] % P, :]
            if kv_dtype == in_dtype:
                assert got.tobytes() == x[r].tobytes()
            else:
                np.testing.assert_array_equal(got, W.as_f32(x[r], in_dtype))
        # every other slot is untouched
        mask = np.ones(kp.shape[0:1] + kp.shape[2:3], bool)
        for r in range(5):
            mask[bt[seq[r], pos[r] // P], pos[r] % P] = False
        assert not kp.transpose(0, 2, 1, 3)[mask].any()


def test_append_rejects_out_of_range():
    x = np.zeros((1, 1, 4), np.float32)
    bt = np.array([[0, -1]], np.int32)
    kp = np.zeros((1, 1, 2, 4), np.float32)
    args = lambda s, p: (x, x, W.F32, np.array([s], np.int32), np.array([p], np.int32), bt, 1, 2, 1, 4,
                         W.F32, 1, 1, kp, kp.copy())
    assert oracle.append(*args(0, 1)) == 0
    assert oracle.append(*args(0, 2)) == -1   # table entry -1
    assert oracle.append(*args(1, 0)) == -1   # no such sequence
    assert oracle.append(*args(0, 4)) == -1   # past max_blocks


def test_bf16_encoder_matches_torch_rne():
    bits = np.concatenate([
        RNG.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32),
        # exact ties (low half 0x8000) with even and odd kept parts, and neighbours
        (RNG.integers(0, 2**16, size=20_000, dtype=np.uint32) << 16) | 0x8000,
        (RNG.integers(0, 2**16, size=20_000, dtype=np.uint32) << 16) | 0x7FFF,
        (RNG.integers(0, 2**16, size=20_000, dtype=np.uint32) << 16) | 0x8001,
    ])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_f32(v) for v in x[:5000]], np.uint16)
    np.testing.assert_array_equal(got, ref[:5000])
    # and the vectorised path through append (f32 rows into a bf16 pool)
    n = (x.size // 64) * 64
    xs = np.ascontiguousarray(x[:n].reshape(-1, 1, 64))
    bt = np.arange(xs.shape[0], dtype=np.int32).reshape(1, -1)
    kp = np.zeros((xs.shape[0], 1, 1, 64), np.uint16)
    assert oracle.append(xs, xs, W.F32, np.zeros(xs.shape[0], np.int32), np.arange(xs.shape[0], dtype=np.int32),
                         bt, xs.shape[0], 1, 1, 64, W.BF16, 1, 1, kp, kp.copy()) == 0
    np.testing.assert_array_equal(kp.reshape(-1), ref[:n])


def _e4m3_value_from_definition(code):
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e4m3_decode_every_code():
    for c in range(256):
        got, ref = oracle.e4m3_to_f64(c), _e4m3_value_from_definition(c)
        assert (math.isnan(got) and math.isnan(ref)) or got == ref, c
    assert oracle.e4m3_to_f64(0x7E) == 448.0 and oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6 and oracle.e4m3_to_f64(0x38) == 1.0


def test_e4m3_encode_decode_identity_and_saturation():
    for c in range(256):
        v = oracle.e4m3_to_f64(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_from_f32(v) == c, c
    for big in (448.0, 449.0, 463.9, 464.0, 500.0, 1e30, math.inf):
        assert oracle.e4m3_from_f32(big) == 0x7E and oracle.e4m3_from_f32(-big) == 0xFE
    assert oracle.e4m3_from_f32(math.nan) == 0x7F
    assert oracle.e4m3_from_f32(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_from_f32(3 * 2.0 ** -10) == 0x02      # tie between 1 and 2 -> even (2)
    assert oracle.e4m3_from_f32(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01


def test_e4m3_encoder_matches_torch_in_non_saturating_range():
    """torch's float8_e4m3fn cast rounds to nearest even; inside |x| < 464 it
    needs no saturation, so it must agree with the oracle code for code."""
    hi16 = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    bits = (hi16[:, None] | lows[None, :]).reshape(-1)
    bits = np.concatenate([bits, RNG.integers(0, 2**32, size=300_000, dtype=np.uint64).astype(np.uint32)])
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_f32_array(x)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encoder_is_monotone_and_saturating():
    x = np.sort(np.concatenate([RNG.standard_normal(200_000).astype(np.float32) * 300,
                                np.linspace(-600, 600, 100_001, dtype=np.float32)]))
    codes = oracle.e4m3_from_f32_array(x)
    vals = np.array([oracle.e4m3_to_f64(c) for c in range(256)])[codes]
    assert np.all(np.diff(vals) >= 0)
    assert vals.max() == 448.0 and vals.min() == -448.0


def test_fp8_append_divides_by_scale_in_binary32():
    """enc(x) = e4m3(x / scale) with one IEEE binary32 division."""
    x = RNG.standard_normal(4096).astype(np.float32) * 3
    scale = np.float32(0.0137)
    xs = x.reshape(-1, 1, 64)
    n = xs.shape[0]
    bt = np.arange(n, dtype=np.int32).reshape(1, -1)
    kp = np.zeros((n, 1, 1, 64), np.uint8)
    vp = kp.copy()
    assert oracle.append(xs, xs, W.F32, np.zeros(n, np.int32), np.arange(n, dtype=np.int32), bt, n, 1, 1, 64,
                         W.E4M3, float(scale), float(scale), kp, vp) == 0
    quotient = (x / scale).astype(np.float32)  # numpy float32 division is IEEE binary32
    ref = torch.from_numpy(quotient).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inside = np.abs(quotient) < 464.0  # torch's cast does not saturate; satfinite does
    assert inside.sum() > 3000 and (~inside).sum() > 50
    np.testing.assert_array_equal(kp.reshape(-1)[inside], ref[inside])
    np.testing.assert_array_equal(kp.reshape(-1)[~inside], np.where(quotient[~inside] > 0, 0x7E, 0xFE))


# -------------------------------------------- p7: causal chunk = decode rows ----

def test_chunk_rows_equal_independent_decode_rows():
    rng = np.random.default_rng(41)
    wl, kp, vp, xk, xv, seq, pos = make_case(rng, [80], Hq=4, Hkv=2, D=16, P=8)
    # a chunk: rows of sequence 0 at positions 40..79, all in one call
    n = 40
    q = rng.standard_normal((n, 4, 16)).astype(np.float32)
    args = dict(q_dtype=W.F32, num_q_heads=4, block_tables=wl.block_tables, num_pages=wl.num_pages,
                page_size=8, num_kv_heads=2, head_dim=16, kv_dtype=W.F32, k_scale=1, v_scale=1,
                k_pool=kp, v_pool=vp)
    together = oracle.attention(q, seq_ids=np.zeros(n, np.int32), positions=np.arange(40, 80, dtype=np.int32),
                                **args)
    for i in (0, 17, 39):
        alone = oracle.attention(q[i:i + 1], seq_ids=np.zeros(1, np.int32),
                                 positions=np.array([40 + i], np.int32), **args)
        assert alone.tobytes() == together[i:i + 1].tobytes()
    # and the causal mask: row at position 40 must not see keys 41..79
    wl1 = W.Workload(**{**wl.__dict__, "q": q[:1], "seq_ids": np.zeros(1, np.int32),
                        "positions": np.array([40], np.int32)})
    np.testing.assert_allclose(together[0], brute_force(wl1, xk, xv, seq, pos)[0], rtol=1e-12)


# ----------------------------------------------------- p8: merge algebra ----

def test_split_merge_algebra():
    """Partial (max, sum, acc) triples over fixed key chunks, merged in order,
    reproduce the unsplit softmax-weighted sum (the GPU's split-KV merge)."""
    rng = np.random.default_rng(51)
    L, D = 1000, 32
    s = rng.standard_normal(L) * 3
    V = rng.standard_normal((L, D))
    full = softmax(s) @ V
    for chunk in (1, 7, 128, 999, 1000):
        ms, ls, accs = [], [], []
        for c0 in range(0, L, chunk):
            sc = s[c0:c0 + chunk]
            m = sc.max()
            w = np.exp(sc - m)
            ms.append(m)
            ls.append(w.sum())
            accs.append(w @ V[c0:c0 + chunk])
        M = max(ms)
        lsum, osum = 0.0, np.zeros(D)
        for m, l, a in zip(ms, ls, accs):
            f = math.exp(m - M)
            lsum += f * l
            osum += f * a
        np.testing.assert_allclose(osum / lsum, full, rtol=1e-12, atol=1e-13)


# ------------------------------------- the pages' printed page counts ----

def test_page_counts_printed_for_32_token_pages():
    """'GPU inference engine engineering', 'Batching without running out of
    cache': with 32-token pages a 2,662-token request holds 86 pages once the
    answer is reserved, and its prompt alone needs 84 (ceil(2662/32)); a short
    call of 5 pages holds up to 160 tokens.  The workload's block tables use
    the same arithmetic."""
    assert math.ceil(2662 / 32) == 84 <= 86
    assert math.ceil(5 * 32 / 32) == 5
    wl = W.mixed_step(n_decode=2, ctx_hi=100)
    cs = wl.num_seqs - 1
    assert int((wl.block_tables[cs] >= 0).sum()) == 84


def test_per_head_scales_equal_per_tensor_on_rescaled_inputs():
    """One fp8 scale per kv head.  With power-of-two scales s_h (keys) and t_h
    (values), appending K = s_h * y and V = t_h * z with the per-head scales
    stores the same codes as appending y and z with scale 1; attention then
    equals scale-1 attention with each query head of group h multiplied by s_h,
    times t_h.  A head index mixed up anywhere (encode, key decode, value
    decode) breaks one of the two equalities."""
    rng = np.random.default_rng(12)
    Hkv, G, D, P, npg = 3, 2, 16, 8, 12
    s_h = np.array([2.0 ** -3, 2.0 ** -6, 2.0 ** 1], np.float32)
    t_h = np.array([2.0 ** 2, 2.0 ** -5, 2.0 ** -1], np.float32)
    ctx = [5, 17, 30]
    bt = np.full((3, 4), -1, np.int32)
    bt[0, :1], bt[1, :3], bt[2, :4] = [7], [0, 3, 9], [1, 2, 4, 11]
    seq = np.repeat(np.arange(3, dtype=np.int32), ctx)
    pos = np.concatenate([np.arange(c, dtype=np.int32) for c in ctx])
    y = W.to_bf16_bits(rng.standard_normal((len(seq), Hkv, D)).astype(np.float32) * 40)
    z = W.to_bf16_bits(rng.standard_normal((len(seq), Hkv, D)).astype(np.float32) * 40)
    yf, zf = W.bf16_bits_to_f32(y), W.bf16_bits_to_f32(z)
    x = W.to_bf16_bits(yf * s_h[None, :, None])  # exact: powers of two
    u = W.to_bf16_bits(zf * t_h[None, :, None])
    pools = {}
    for name, (kin, vin, ks, vs) in {"per_head": (x, u, s_h, t_h), "unit": (y, z, 1.0, 1.0)}.items():
        kp = np.zeros((npg, Hkv, P, D), np.uint8)
        vp = np.zeros((npg, Hkv, P, D), np.uint8)
        assert oracle.append(kin, vin, W.BF16, seq, pos, bt, npg, P, Hkv, D, W.E4M3, ks, vs, kp, vp) == 0
        pools[name] = (kp, vp)
    assert pools["per_head"][0].tobytes() == pools["unit"][0].tobytes()
    assert pools["per_head"][1].tobytes() == pools["unit"][1].tobytes()
    q = rng.standard_normal((3, Hkv * G, D)).astype(np.float32)
    qs = (q * np.repeat(s_h, G)[None, :, None]).astype(np.float32)
    rows = np.arange(3, dtype=np.int32)
    last = np.array(ctx, np.int32) - 1
    kp, vp = pools["per_head"]
    a = oracle.attention(q, W.F32, Hkv * G, rows, last, bt, npg, P, Hkv, D, W.E4M3, s_h, t_h, kp, vp)
    b = oracle.attention(qs, W.F32, Hkv * G, rows, last, bt, npg, P, Hkv, D, W.E4M3, 1.0, 1.0, kp, vp)
    np.testing.assert_allclose(a, b * np.repeat(t_h, G)[None, :, None], rtol=1e-13, atol=0)
    # and the per-head path with equal scales is the per-tensor path, bit for bit
    c = oracle.attention(q, W.F32, Hkv * G, rows, last, bt, npg, P, Hkv, D, W.E4M3, np.full(Hkv, 0.5, np.float32),
                         np.full(Hkv, 0.25, np.float32), kp, vp)
    d = oracle.attention(q, W.F32, Hkv * G, rows, last, bt, npg, P, Hkv, D, W.E4M3, 0.5, 0.25, kp, vp)
    assert c.tobytes() == d.tobytes()
