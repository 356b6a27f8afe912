"""Oracle-side setup for the parity tests: the CPU oracle's own pools, built
by its own append from the workload's inputs, and its attention output."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W


def oracle_pools(wl: W.Workload, rows_of_seqs=None, include_step=True):
    """Oracle append of the history rows (optionally only those of some
    sequences), then of the step's rows.  Returns (k_pool, v_pool)."""
    return oracle.workload_pools(wl, rows_of_seqs=rows_of_seqs, include_step=include_step)


def oracle_out(wl: W.Workload, kp, vp, rows=None, n_threads=None):
    """float64 [n_rows or len(rows), Hq, D] attention of the chosen rows."""
    idx = np.arange(wl.n_rows) if rows is None else np.asarray(rows)
    return oracle.attention(wl.q[idx], wl.q_dtype, wl.Hq, wl.seq_ids[idx], wl.positions[idx], wl.block_tables,
                            wl.num_pages, wl.P, wl.Hkv, wl.D, wl.kv_dtype, wl.k_scale, wl.v_scale, kp, vp,
                            softmax_scale=wl.softmax_scale,
                            n_threads=n_threads or oracle.host_cores())


def tolerances(wl: W.Workload):
    """(abs, rel): f32 K/V 1e-5 / 1e-5; bf16 and fp8 K/V 2e-3 / 1e-2.  An
    element passes if it is within EITHER bound (output rounding to bf16 alone
    is up to 2^-9 relative, which exceeds 2e-3 absolute once |out| > 1)."""
    return (1e-5, 1e-5) if wl.kv_dtype == W.F32 else (2e-3, 1e-2)


def assert_close(got: np.ndarray, ref: np.ndarray, wl: W.Workload, what=""):
    atol, rtol = tolerances(wl)
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    ok = (err <= atol) | (err <= rtol * np.abs(ref))
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} elements out of tolerance "
                             f"(first at {i}: got {got[i]!r} ref {ref[i]!r}); max abs {err.max():.3e}")
    return float(err.max()), float((err / np.maximum(np.abs(ref), 1e-30)).max())
