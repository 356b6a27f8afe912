"""The host page allocator with admission (pa_pages_*), on the CPU: the page
count it predicts, typed refusals with their numbers, all-or-nothing
admission, release and reuse, reference-counted prefix sharing, invariants
under random operation sequences, and block tables it writes driving the
oracle to the same result as un-paged attention."""
import math

import numpy as np
import pytest

import oracle
import paged_kv_continuous_pa_gb300 as pa
import workloads as W


@pytest.fixture(scope="module", autouse=True)
def lib():
    pa.load()


def snapshot(a: pa.Pages):
    return a.free_count(), a.block_tables.copy(), [a.refcount(i) for i in range(a.block_tables.size)]


def test_pages_needed_is_the_ceiling():
    for P in (1, 16, 32, 64):
        for prompt in (0, 1, 31, 32, 33, 1000):
            for new in (0, 1, 63, 64, 65):
                assert pa.pages_needed(P, prompt, new) == math.ceil((prompt + new) / P)
    assert pa.pages_needed(0, 1, 1) == -1 and pa.pages_needed(32, -1, 0) == -1


def test_admission_until_exhausted_then_typed_refusal():
    a = pa.Pages(num_pages=20, page_size=32, num_seqs=8, max_blocks=16)
    got = []
    for s, (prompt, new) in enumerate([(100, 28), (32, 0), (200, 56), (1, 1)]):  # 4 + 1 + 8 + 1 pages
        st, info = a.admit(s, prompt, new)
        assert st == pa.PA_OK and info.reason == pa.PA_ADMIT_OK
        n = pa.pages_needed(32, prompt, new)
        assert info.pages_needed == n and info.tokens == prompt + new and info.max_tokens == 16 * 32
        row = a.block_tables[s]
        assert (row[:n] >= 0).all() and (row[n:] == -1).all()
        got.extend(row[:n].tolist())
    assert got == list(range(14))  # a fresh allocator hands out the lowest ids first
    assert a.free_count() == 6
    before = snapshot(a)
    st, info = a.admit(4, 150, 60)  # 7 pages, 6 free
    assert st == pa.PA_ERR_NO_PAGES and info.reason == pa.PA_ADMIT_NO_PAGES
    assert (info.pages_needed, info.pages_free, info.tokens) == (7, 6, 210)
    assert "needs 7 new pages" in pa.last_error() and "6 are free" in pa.last_error()
    after = snapshot(a)
    assert before[0] == after[0] and (before[1] == after[1]).all() and before[2] == after[2]
    st, _ = a.admit(4, 150, 42)  # 6 pages fit exactly
    assert st == pa.PA_OK and a.free_count() == 0


@pytest.mark.parametrize("case", ["too_long", "in_use", "bad_seq", "negative", "bad_parent", "prefix_past_prompt"])
def test_other_refusals_change_nothing(case):
    a = pa.Pages(num_pages=40, page_size=16, num_seqs=4, max_blocks=8)
    assert a.admit(0, 50, 10)[0] == pa.PA_OK
    before = snapshot(a)
    args, reason = {
        "too_long": ((1, 100, 29), pa.PA_ADMIT_TOO_LONG),       # 129 > 8 * 16
        "in_use": ((0, 10, 10), pa.PA_ADMIT_SEQ_IN_USE),
        "bad_seq": ((4, 10, 10), pa.PA_ADMIT_BAD_ARG),
        "negative": ((1, -1, 10), pa.PA_ADMIT_BAD_ARG),
        "bad_parent": ((1, 40, 10, 2, 32), pa.PA_ADMIT_BAD_ARG),  # slot 2 not admitted
        "prefix_past_prompt": ((1, 40, 10, 0, 48), pa.PA_ADMIT_BAD_ARG),
    }[case]
    st, info = a.admit(*args)
    assert st == pa.PA_ERR_INVALID_ARG and info.reason == reason
    after = snapshot(a)
    assert before[0] == after[0] and (before[1] == after[1]).all() and before[2] == after[2]
    if case == "too_long":
        assert (info.tokens, info.max_tokens) == (129, 128)


def test_release_returns_pages_and_readmission_gets_the_same_ones():
    a = pa.Pages(num_pages=12, page_size=32, num_seqs=3, max_blocks=8)
    assert a.admit(0, 70, 10)[0] == pa.PA_OK   # 3 pages
    assert a.admit(1, 100, 0)[0] == pa.PA_OK   # 4 pages
    row1 = a.block_tables[1].copy()
    a.release(1)
    assert (a.block_tables[1] == -1).all() and a.free_count() == 9
    assert a.admit(1, 100, 0)[0] == pa.PA_OK
    assert (a.block_tables[1] == row1).all()
    with pytest.raises(pa.PaError):
        a.release(2)  # holds nothing


def test_prefix_pages_are_shared_and_reference_counted():
    P = 32
    a = pa.Pages(num_pages=30, page_size=P, num_seqs=4, max_blocks=10)
    assert a.admit(0, 100, 20)[0] == pa.PA_OK  # 4 pages
    parent = a.block_tables[0].copy()
    st, info = a.admit(1, 150, 10, prefix_parent=0, prefix_tokens=90)  # 90 tokens: 2 whole pages shared
    assert st == pa.PA_OK and info.pages_shared == 2 and info.pages_needed == 5 - 2
    child = a.block_tables[1]
    assert (child[:2] == parent[:2]).all() and not set(child[2:5].tolist()) & set(parent[:4].tolist())
    assert [a.refcount(int(p)) for p in parent[:4]] == [2, 2, 1, 1]
    free = a.free_count()
    a.release(0)  # the shared pages stay held by the child
    assert a.free_count() == free + 2 and [a.refcount(int(p)) for p in parent[:2]] == [1, 1]
    a.release(1)
    assert a.free_count() == 30 and all(a.refcount(i) == 0 for i in range(30))


def test_random_operations_keep_the_invariants():
    rng = np.random.default_rng(7)
    P, npg, nseq, mb = 16, 64, 12, 12
    a = pa.Pages(npg, P, nseq, mb)
    admitted = {}  # seq -> (tokens, parent, shared)
    for _ in range(3000):
        s = int(rng.integers(nseq))
        if s in admitted and rng.random() < 0.5:
            a.release(s)
            del admitted[s]
        else:
            prompt, new = int(rng.integers(0, 120)), int(rng.integers(0, 80))
            parent, pref = -1, 0
            if admitted and rng.random() < 0.4:
                parent = int(rng.choice(list(admitted)))
                pref = int(rng.integers(0, prompt + 1))
            before = snapshot(a)
            st, info = a.admit(s, prompt, new, parent, pref)
            if st == pa.PA_OK:
                shared = min(pref // P, int((a.block_tables[parent] >= 0).sum())) if parent >= 0 else 0
                admitted[s] = (prompt + new, parent, shared)
            else:
                after = snapshot(a)
                assert before[0] == after[0] and (before[1] == after[1]).all() and before[2] == after[2]
                if st == pa.PA_ERR_NO_PAGES:
                    assert info.pages_needed > info.pages_free == a.free_count()
        # invariants
        refs = np.zeros(npg, np.int64)
        for q, (tok, _, _) in admitted.items():
            row = a.block_tables[q]
            n = math.ceil(tok / P)
            assert (row[:n] >= 0).all() and (row[n:] == -1).all()
            assert len(set(row[:n].tolist())) == n
            refs[row[:n]] += 1
        for q in set(range(nseq)) - set(admitted):
            assert (a.block_tables[q] == -1).all()
        assert [a.refcount(i) for i in range(npg)] == refs.tolist()
        assert a.free_count() == int((refs == 0).sum())


def test_allocator_tables_drive_the_oracle_like_unpaged_attention():
    """Sequences admitted through the allocator (one sharing a parent's prefix
    pages), their prompts appended through the tables by the oracle, then one
    decode row each: equal to float64 attention over the un-paged rows."""
    rng = np.random.default_rng(3)
    P, Hkv, G, D = 16, 2, 2, 64
    a = pa.Pages(num_pages=64, page_size=P, num_seqs=3, max_blocks=16)
    prompts = [70, 41, 90]
    assert a.admit(0, prompts[0], 20)[0] == pa.PA_OK
    assert a.admit(1, prompts[1], 20)[0] == pa.PA_OK
    assert a.admit(2, prompts[2], 20, prefix_parent=0, prefix_tokens=48)[0] == pa.PA_OK  # 3 shared pages
    bt = a.block_tables
    keys = [rng.standard_normal((L + 1, Hkv, D)).astype(np.float32) for L in prompts]
    vals = [rng.standard_normal((L + 1, Hkv, D)).astype(np.float32) for L in prompts]
    keys[2][:48], vals[2][:48] = keys[0][:48], vals[0][:48]  # the shared prefix holds the parent's rows
    kp = np.full((64, Hkv, P, D), np.nan, np.float32)
    vp = kp.copy()
    for s, L in enumerate(prompts):
        first = 48 if s == 2 else 0  # shared pages are never appended again
        pos = np.arange(first, L + 1, dtype=np.int32)
        st = oracle.append(keys[s][first:], vals[s][first:], W.F32, np.full(len(pos), s, np.int32), pos, bt, 64, P, Hkv,
                           D, W.F32, 1.0, 1.0, kp, vp)
        assert st == 0
    q = rng.standard_normal((3, Hkv * G, D)).astype(np.float32)
    out = oracle.attention(q, W.F32, Hkv * G, np.arange(3, dtype=np.int32), np.array(prompts, np.int32), bt, 64, P,
                           Hkv, D, W.F32, 1.0, 1.0, kp, vp, n_threads=1)
    for s in range(3):
        for g in range(Hkv * G):
            k, v = keys[s][:, g // G].astype(np.float64), vals[s][:, g // G].astype(np.float64)
            sc = k @ q[s, g].astype(np.float64) / np.sqrt(D)
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(out[s, g], (w / w.sum()) @ v, rtol=1e-12, atol=1e-12)
