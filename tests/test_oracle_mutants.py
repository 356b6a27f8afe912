"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in test_oracle.py catch every one: a dropped term, a wrong sign, a
wrong index, a transposed operand, a wrong tie rule.  The copy is compiled
into a temporary directory; the real oracle is never modified."""
import os
import subprocess

import numpy as np
import pytest

import oracle

import test_oracle as T

# (name, original text, mutated text); each original occurs exactly once
MUTANTS = [
    ("own token dropped", "int64_t L = (int64_t)p + 1;", "int64_t L = (int64_t)p;"),
    ("kv head by modulo", "int h = g / G;", "int h = g % H;"),
    ("no normalisation", "a->out[qoff + d] = acc[d] / z;", "a->out[qoff + d] = acc[d];"),
    ("softmax scale dropped", "score[t] = a->softmax_scale * dot;", "score[t] = dot;"),
    ("exponent sign flipped", "double w = exp(score[t] - m);", "double w = exp(m - score[t]);"),
    ("query head index", "int64_t qoff = ((int64_t)r * Hq + g) * D;",
     "int64_t qoff = ((int64_t)r * Hq + h) * D;"),
    ("value from the key pool", "acc[d] += w * load_pool(a->v_pool,", "acc[d] += w * load_pool(a->k_pool,"),
    ("slot and head transposed in key reads",
     "int64_t base = (((int64_t)page_of[t / P] * H + h) * P + t % P) * D;\n                double dot",
     "int64_t base = (((int64_t)page_of[t / P] * P + t % P) * H + h) * D;\n                double dot"),
    ("append page index by modulo", "block_tables[(int64_t)s * max_blocks + p / P];",
     "block_tables[(int64_t)s * max_blocks + p % P];"),
    ("fp8 ties away from zero", "code = (lo & 1) ? hi : lo;", "code = hi;"),
    ("bf16 ties away from zero", "u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    ("fp8 subnormal exponent", "v = ldexp((double)m / 8.0, 1 - 7);", "v = ldexp((double)m / 8.0, -7);"),
    ("fp8 scale not applied on decode", "oracle_e4m3_to_f64(((const uint8_t *)pool)[i]) * (double)scale;",
     "oracle_e4m3_to_f64(((const uint8_t *)pool)[i]);"),
    ("fp8 encode multiplies by the scale", "load_as_f32(src, in_dtype, j) / scale;",
     "load_as_f32(src, in_dtype, j) * scale;"),
    ("overflow to NaN instead of saturating", "if (a >= 448.0)\n        return sign | 0x7e;",
     "if (a >= 448.0)\n        return sign | 0x7f;"),
    ("per-head key scale of the wrong head on append",
     "store_pool(k_pool, kv_dtype, dst, k_new, in_dtype, src, k_scales[h])",
     "store_pool(k_pool, kv_dtype, dst, k_new, in_dtype, src, k_scales[(h + 1) % H])"),
    ("per-head value scale of the wrong head on decode",
     "load_pool(a->v_pool, a->kv_dtype, base + d, a->v_scales[h]);",
     "load_pool(a->v_pool, a->kv_dtype, base + d, a->v_scales[0]);"),
    ("per-head key scale of the wrong head on decode",
     "load_pool(a->k_pool, a->kv_dtype, base + d, a->k_scales[h]);",
     "load_pool(a->k_pool, a->kv_dtype, base + d, a->k_scales[H - 1 - h]);"),
]

PINS = [
    lambda: T.test_matches_contiguous_brute_force_f32(64, 2, 4),
    lambda: T.test_matches_contiguous_brute_force_f32(4, 1, 1),
    lambda: T.test_matches_brute_force_storage_dtypes(T.W.E4M3, T.W.BF16),
    lambda: T.test_identical_keys_give_mean_of_values(),
    lambda: T.test_single_position_returns_its_value_exactly(T.W.E4M3),
    lambda: T.test_hand_worked_two_token_case(),
    lambda: T.test_append_roundtrip_and_page_boundary(),
    lambda: T.test_bf16_encoder_matches_torch_rne(),
    lambda: T.test_e4m3_decode_every_code(),
    lambda: T.test_e4m3_encode_decode_identity_and_saturation(),
    lambda: T.test_e4m3_encoder_matches_torch_in_non_saturating_range(),
    lambda: T.test_fp8_append_divides_by_scale_in_binary32(),
    lambda: T.test_per_head_scales_equal_per_tensor_on_rescaled_inputs(),
]


def _build_mutant(tmp_path, orig, mutated):
    src = open(os.path.join(oracle.HERE, "oracle.c")).read()
    assert src.count(orig) == 1, orig
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(orig, mutated))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                    str(path), "-o", str(so), "-lm"], check=True)
    return oracle.load(str(so))


def test_pins_pass_on_the_real_oracle():
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name,orig,mutated", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, mutated, monkeypatch):
    mutant = _build_mutant(tmp_path, orig, mutated)
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = []
    with np.errstate(all="ignore"):
        for i, pin in enumerate(PINS):
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(i)
    assert caught, f"mutant '{name}' survived every pin"
