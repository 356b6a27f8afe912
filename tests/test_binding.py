"""The Python binding rejects tensors whose dtype or shape the C ABI cannot
see (int32 index arrays, q / out / k_new / v_new against the pool's shape)
before any pointer is passed; checked on the CPU with a stand-in pool."""
import types

import pytest
import torch

import paged_kv_continuous_pa_gb300 as pa

POOL = types.SimpleNamespace(head_dim=64, num_kv_heads=2, handle=None)
N, HQ = 3, 4


def good():
    return dict(q=torch.zeros(N, HQ, 64, dtype=torch.bfloat16), seq_ids=torch.zeros(N, dtype=torch.int32),
                positions=torch.zeros(N, dtype=torch.int32), block_tables=torch.zeros(2, 5, dtype=torch.int32),
                out=torch.zeros(N, HQ, 64, dtype=torch.bfloat16), status=torch.zeros(1, dtype=torch.int32),
                k_new=torch.zeros(N, 2, 64, dtype=torch.bfloat16), v_new=torch.zeros(N, 2, 64, dtype=torch.bfloat16))


def call_attention(a):
    return pa.attention(POOL, a["q"], a["seq_ids"], a["positions"], a["block_tables"], a["out"], status=a["status"])


def call_step(a):
    return pa.step(POOL, a["q"], a["k_new"], a["v_new"], a["seq_ids"], a["positions"], a["block_tables"], a["out"],
                   status=a["status"])


def call_append(a):
    return pa.append_kv(POOL, a["k_new"], a["v_new"], a["seq_ids"], a["positions"], a["block_tables"],
                        status=a["status"])


@pytest.mark.parametrize("call", [call_attention, call_step, call_append])
@pytest.mark.parametrize("name", ["seq_ids", "positions", "block_tables", "status"])
def test_index_arrays_must_be_int32(call, name):
    a = good()
    a[name] = a[name].to(torch.int64)
    with pytest.raises(TypeError, match=name):
        call(a)


@pytest.mark.parametrize("case", ["positions_rows", "block_tables_1d", "q_head_dim", "q_rows", "out_shape", "out_dtype"])
def test_attention_shapes(case):
    a = good()
    if case == "positions_rows":
        a["positions"] = torch.zeros(N + 1, dtype=torch.int32)
    elif case == "block_tables_1d":
        a["block_tables"] = torch.zeros(10, dtype=torch.int32)
    elif case == "q_head_dim":
        a["q"] = torch.zeros(N, HQ, 128, dtype=torch.bfloat16)
        a["out"] = torch.zeros(N, HQ, 128, dtype=torch.bfloat16)
    elif case == "q_rows":
        a["q"] = torch.zeros(N + 1, HQ, 64, dtype=torch.bfloat16)
        a["out"] = torch.zeros(N + 1, HQ, 64, dtype=torch.bfloat16)
    elif case == "out_shape":
        a["out"] = torch.zeros(N, HQ, 32, dtype=torch.bfloat16)
    elif case == "out_dtype":
        a["out"] = torch.zeros(N, HQ, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        call_attention(a)


@pytest.mark.parametrize("case", ["k_heads", "v_dim", "kv_rows", "kv_dtypes"])
@pytest.mark.parametrize("call", [call_step, call_append])
def test_new_rows_match_the_pool(call, case):
    a = good()
    if case == "k_heads":
        a["k_new"] = torch.zeros(N, 4, 64, dtype=torch.bfloat16)
    elif case == "v_dim":
        a["v_new"] = torch.zeros(N, 2, 128, dtype=torch.bfloat16)
    elif case == "kv_rows":
        a["k_new"] = torch.zeros(N + 2, 2, 64, dtype=torch.bfloat16)
        a["v_new"] = torch.zeros(N + 2, 2, 64, dtype=torch.bfloat16)
    elif case == "kv_dtypes":
        a["v_new"] = torch.zeros(N, 2, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        call(a)


def test_valid_arguments_reach_the_device_check():
    """Everything checkable on the host passes; the first refusal is that the tensors are not on a GPU."""
    with pytest.raises(ValueError, match="CUDA"):
        call_attention(good())
