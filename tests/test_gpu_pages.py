"""Block tables from the host page allocator (pa_pages_*), some sequences
sharing a parent's prefix pages, driving the GPU step (pa_step) against the
oracle: pool bytes identical, outputs within tolerance."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


def allocator_workload(seed, Hq, Hkv, D, P, kv_dtype):
    rng = np.random.default_rng(seed)
    n_seqs, num_pages, max_blocks = 10, 160, 16
    a = pa.Pages(num_pages, P, n_seqs, max_blocks)
    prompts = rng.integers(1, max_blocks * P - 64, size=n_seqs)
    parents = {}
    for s in range(n_seqs):
        parent, pref = -1, 0
        if s >= 4 and rng.random() < 0.6:  # share a prefix with one of the first four
            parent = int(rng.integers(4))
            pref = int(min(prompts[s], prompts[parent], rng.integers(P, 5 * P)))
        st, info = a.admit(s, int(prompts[s]), 32, parent, pref)
        assert st == pa.PA_OK, pa.last_error()
        parents[s] = (parent, pref, info.pages_shared)
    in_dtype = kv_dtype if kv_dtype != W.E4M3 else W.BF16
    keys = [rng.standard_normal((int(L) + 1, Hkv, D)).astype(np.float32) for L in prompts]
    vals = [rng.standard_normal((int(L) + 1, Hkv, D)).astype(np.float32) for L in prompts]
    hs, hp, hk, hv = [], [], [], []
    for s in range(n_seqs):
        parent, pref, shared = parents[s]
        if parent >= 0:  # the prefix tokens hold the parent's rows
            keys[s][:pref], vals[s][:pref] = keys[parent][:pref], vals[parent][:pref]
        first = shared * P  # whole shared pages are the parent's: never appended again
        L = int(prompts[s])
        hs.append(np.full(L - first, s, np.int32))
        hp.append(np.arange(first, L, dtype=np.int32))
        hk.append(keys[s][first:L])
        hv.append(vals[s][first:L])
    wl = W.Workload(name="pages", Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=kv_dtype, in_dtype=in_dtype, q_dtype=W.BF16,
                    num_pages=num_pages, block_tables=a.block_tables.copy(), hist_seq=np.concatenate(hs),
                    hist_pos=np.concatenate(hp), hist_k=W._cast(np.concatenate(hk), in_dtype),
                    hist_v=W._cast(np.concatenate(hv), in_dtype), seq_ids=np.arange(n_seqs, dtype=np.int32),
                    positions=prompts.astype(np.int32),
                    q=W._cast(rng.standard_normal((n_seqs, Hq, D)).astype(np.float32), W.BF16),
                    k_new=W._cast(np.stack([keys[s][int(prompts[s])] for s in range(n_seqs)]), in_dtype),
                    v_new=W._cast(np.stack([vals[s][int(prompts[s])] for s in range(n_seqs)]), in_dtype),
                    description="allocator tables")
    if kv_dtype == W.E4M3:
        wl.k_scale, wl.v_scale = 0.0123, 0.0101
    return wl


@pytest.mark.parametrize("shape", ["bf16_g2", "fp8_g7"])
def test_allocator_tables_through_the_gpu_step(shape):
    Hq, Hkv, kv = {"bf16_g2": (16, 8, W.BF16), "fp8_g7": (28, 4, W.E4M3)}[shape]
    wl = allocator_workload(11, Hq, Hkv, 128, 32, kv)
    st = pa_setup.upload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    assert pa_setup.to_numpy(st.k_pool).tobytes() == kp.tobytes()
    assert pa_setup.to_numpy(st.v_pool).tobytes() == vp.tobytes()
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, shape)
