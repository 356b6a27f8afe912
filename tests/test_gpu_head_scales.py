"""One fp8 scale per kv head (pa_pool_set_head_scales) on the GPU against the
oracle with the same per-head scales: pool bytes identical, outputs within
tolerance, on the tensor-core units (D 128, bf16 q) and the SIMT units (D 64,
and f32 queries); and per-head scales that are all equal give the per-tensor
bits."""
import numpy as np
import pytest
import torch

import pa_setup
import paged_kv_continuous_pa_gb300 as pa
import workloads as W
from ref import assert_close, oracle_out, oracle_pools

pytestmark = pytest.mark.gpu


def head_scaled(seed, Hq, Hkv, D, q_dtype):
    ctx = [1, 31, 33, 64, 300, 700]
    wl = W._decode_workload("hs", seed, ctx, Hq, Hkv, D, 32, W.E4M3, q_dtype, max_ctx=704, spare_pages=4,
                            description="per-head fp8 scales")
    # kv head h holds values about 2^h times larger, its scales follow
    f = (2.0 ** np.arange(Hkv)).astype(np.float32)
    for name in ("hist_k", "hist_v", "k_new", "v_new"):
        x = W.as_f32(getattr(wl, name), wl.in_dtype) * f[None, :, None]
        setattr(wl, name, W._cast(x, wl.in_dtype))
    amax_k = np.maximum(np.abs(W.as_f32(wl.hist_k, wl.in_dtype)).max(axis=(0, 2)),
                        np.abs(W.as_f32(wl.k_new, wl.in_dtype)).max(axis=(0, 2)))
    amax_v = np.maximum(np.abs(W.as_f32(wl.hist_v, wl.in_dtype)).max(axis=(0, 2)),
                        np.abs(W.as_f32(wl.v_new, wl.in_dtype)).max(axis=(0, 2)))
    wl.k_scale = (amax_k.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    wl.v_scale = (amax_v.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    return wl


@pytest.mark.parametrize("shape", ["mma_d128_g7", "mma_d128_g2", "simt_d64_g4", "simt_f32q_g7"])
def test_per_head_scales_match_oracle(shape):
    Hq, Hkv, D, qd = {"mma_d128_g7": (28, 4, 128, W.BF16), "mma_d128_g2": (16, 8, 128, W.BF16),
                      "simt_d64_g4": (16, 4, 64, W.BF16), "simt_f32q_g7": (28, 4, 128, W.F32)}[shape]
    wl = head_scaled(41, Hq, Hkv, D, qd)
    st = pa_setup.upload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    assert pa_setup.to_numpy(st.k_pool).tobytes() == kp.tobytes()
    assert pa_setup.to_numpy(st.v_pool).tobytes() == vp.tobytes()
    got = pa_setup.to_numpy(st.out)
    got = got.astype(np.float64) if qd == W.F32 else W.bf16_bits_to_f32(got).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, shape)


def test_equal_head_scales_give_per_tensor_bits():
    wl = head_scaled(42, 28, 4, 128, W.BF16)
    s_k, s_v = float(wl.k_scale.max()), float(wl.v_scale.max())
    outs = []
    for ks, vs in ((s_k, s_v), (np.full(4, s_k, np.float32), np.full(4, s_v, np.float32))):
        wl.k_scale, wl.v_scale = ks, vs
        st = pa_setup.upload(wl)
        st.step()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        outs.append((st.k_pool.view(torch.uint8).clone(), st.out.view(torch.int16).clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("D", [128, 64])
def test_sixty_four_kv_heads_each_with_its_scale(D):
    """The largest per-head table (64 kv heads, one query head each): every head's
    scale is its own, on the tensor-core units (D 128) and the SIMT units (D 64).
    The values keep unit scale (the tolerance's absolute part is stated for
    those); the scales differ by head, from amax / 448 up to 4.5 times that, so
    a head read with another head's scale is off by their ratio."""
    Hkv = 64
    wl = W._decode_workload("hs64", 70 + D, [1, 31, 33, 64, 300], Hkv, Hkv, D, 32, W.E4M3, W.BF16, max_ctx=320,
                            spare_pages=4, description="64 per-head fp8 scales")
    f = (1.0 + 0.5 * (np.arange(Hkv) % 8)).astype(np.float32)
    amax_k = max(np.abs(W.as_f32(wl.hist_k, wl.in_dtype)).max(), np.abs(W.as_f32(wl.k_new, wl.in_dtype)).max())
    amax_v = max(np.abs(W.as_f32(wl.hist_v, wl.in_dtype)).max(), np.abs(W.as_f32(wl.v_new, wl.in_dtype)).max())
    wl.k_scale = (np.float32(amax_k) / np.float32(448.0) * f).astype(np.float32)
    wl.v_scale = (np.float32(amax_v) / np.float32(448.0) * f).astype(np.float32)
    st = pa_setup.upload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    kp, vp = oracle_pools(wl)
    assert pa_setup.to_numpy(st.k_pool).tobytes() == kp.tobytes()
    assert pa_setup.to_numpy(st.v_pool).tobytes() == vp.tobytes()
    got = W.bf16_bits_to_f32(pa_setup.to_numpy(st.out)).astype(np.float64)
    assert_close(got, oracle_out(wl, kp, vp), wl, f"64 heads D{D}")
