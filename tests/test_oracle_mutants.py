"""Planted mistakes: each mutant of the oracle source (a dropped term, a wrong
sign, index or operand, a changed constant) is compiled on the CPU and must
fail at least one of the pins the oracle is held to.  The unmodified source
must pass all of them."""
import pytest

import oracle
import test_oracle_attention as ta
import test_oracle_codec as tc
import test_oracle_fp16 as tf
import test_oracle_nvfp4 as tn

Q4, Q8, Q4_32, NV = oracle.Q4_G64, oracle.Q8_0, oracle.Q4_G32, oracle.NVFP4

PINS = [
    ("golden q4", lambda: tc.test_golden_rows("q4g64_two_groups.txt", Q4)),
    ("golden q8", lambda: tc.test_golden_rows("q8_0_two_groups.txt", Q8)),
    ("golden q4 g32", lambda: tc.test_golden_rows("q4g32_two_groups.txt", Q4_32)),
    ("fp16 edges", tf.test_f32_to_f16_edge_classes),
    ("fp16 dense", tf.test_f32_to_f16_half_range_dense),
    ("brute force q4", lambda: tc.test_brute_force_nearest_code(Q4)),
    ("scale rule q4", lambda: tc.test_scale_rule_and_roundtrip_bound(Q4)),
    ("dequant exact", tc.test_dequant_exact_in_fp64),
    ("append", tc.test_append_positions_and_error_bit),
    ("sdpa q4/q4 n_q=3", lambda: ta.test_matches_torch_sdpa_float64(Q4, Q4, 3, 64)),
    ("sdpa q8/q4", lambda: ta.test_matches_torch_sdpa_float64(Q8, Q4, 1, 128)),
    ("split/merge", lambda: ta.test_split_then_merge_equals_unsplit(3)),
    ("merge closed forms", ta.test_merge_closed_forms),
    ("fraction brute force", lambda: ta.test_exact_rational_brute_force(5)),
    ("golden nvfp4", tn.test_golden_row),
    ("e2m1 binade", tn.test_e2m1_encode_matches_binade_rounding),
    ("e2m1 ties", tn.test_e2m1_ties_and_signed_zero),
    ("e4m3 binade", tn.test_e4m3_encode_matches_binade_rounding_and_saturates),
    ("nvfp4 rule", lambda: tn.test_quantize_matches_the_rule_written_another_way("mixed")),
    ("nvfp4 bound", tn.test_roundtrip_bound_and_exact_dequant),
    ("nvfp4 special", tn.test_special_blocks),
]
if tn.HAS_F8:
    PINS += [("e4m3 torch decode", tn.test_e4m3_decode_matches_torch),
             ("e4m3 torch encode", tn.test_e4m3_encode_matches_torch_in_range)]

MUTANTS = {
    "nibble_order": ("if (v & 1) qr[v >> 1]", "if (!(v & 1)) qr[v >> 1]"),
    "nibble_sign": ("return nib >= 8 ? nib - 16 : nib;", "return nib >= 8 ? nib - 8 : nib;"),
    "scale_divisor": ("float s = amax / (float)qmax;", "float s = amax / (float)(qmax + 1);"),
    "round_half_away": ("float r = nearbyintf(x / d);", "float r = roundf(x / d);"),
    "no_saturation": ("if (d == 0x7C00u) d = 0x7BFFu;", ""),
    "q8_group": ("codec == ORC_NVFP4 ? 16 : 32; }", "codec == ORC_NVFP4 ? 16 : 64; }"),
    "q4_g32_group": ("static int orc_group(int codec) { return codec == ORC_Q4 ? 64 :",
                     "static int orc_group(int codec) { return (codec == ORC_Q4 || codec == ORC_Q4_32) ? 64 :"),
    "nvfp4_scale_divisor": ("uint8_t sb = orc_f32_to_e4m3(amax / 6.0f);", "uint8_t sb = orc_f32_to_e4m3(amax / 7.0f);"),
    "fp8_ties_up": ("if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {", "if (d <= bd) {"),
    "fp8_no_saturation": ("    if (a >= decode((uint8_t)(n_codes - 1))) return n_codes - 1;\n", ""),
    "e4m3_bias": ("else v = (1.0f + (float)m / 8.0f) * ldexpf(1.0f, e - 7);",
                  "else v = (1.0f + (float)m / 8.0f) * ldexpf(1.0f, e - 8);"),
    "e2m1_zero_sign_dropped": ("return (uint8_t)(c | (signbit(f) ? 8 : 0));",
                               "return (uint8_t)(c | (c != 0 && signbit(f) ? 8 : 0));"),
    "nvfp4_zero_scale": ("c[i] = (d == 0.0f) ? 0 : orc_f32_to_e2m1(x[i] / d);", "c[i] = orc_f32_to_e2m1(x[i] / d);"),
    "f16_truncates": ("if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;", ""),
    "f16_subnormal_shift": ("uint32_t shift = 126u - e;", "uint32_t shift = 127u - e;"),
    "gqa_mapping": ("int r = i * G + j, h = kh * G + j;", "int r = i * G + j, h = kh + j * a->n_kv_heads;"),
    "causal_off_by_one": ("int64_t n = (int64_t)kv_len - n_q + i + 1;", "int64_t n = (int64_t)kv_len - n_q + i;"),
    "dropped_scale": ("z[r * span + t] = acc * a->scale;", "z[r * span + t] = acc;"),
    "transposed_operand": ("acc += qd[r * D + d] * (double)kr[d];", "acc += qd[r * D + d] * (double)kr[D - 1 - d];"),
    "k_read_as_v": ("orc_dequantize(a->v_codec, a->v_qs + row * vrb", "orc_dequantize(a->v_codec, a->k_qs + row * vrb"),
    "lse_without_max": ("lse[(int64_t)r * lse_row_stride] = m[r] + log(l[r]);",
                        "lse[(int64_t)r * lse_row_stride] = log(l[r]);"),
    "sum_overwritten": ("l[r] += z[r * span + t];", "l[r] = z[r * span + t];"),
    "merge_unweighted": ("double w = exp(ls - M);", "double w = 1.0;"),
    "append_position": ("* capacity + pos0[s] + i;", "* capacity + pos0[s];"),
}


def _run_pins():
    failed = []
    for name, pin in PINS:
        try:
            pin()
        except Exception:                 # an assertion or a shape/validity error
            failed.append(name)
    return failed


def test_unmodified_source_passes_every_pin(tmp_path):
    lib = oracle.compile_source(oracle.source(), str(tmp_path / "orig.so"))
    with oracle.using_library(lib):
        assert _run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    find, repl = MUTANTS[name]
    src = oracle.source()
    assert src.count(find) == 1, f"mutation anchor for {name} not unique"
    lib = oracle.compile_source(src.replace(find, repl), str(tmp_path / f"mut_{name}.so"))
    with oracle.using_library(lib):
        failed = _run_pins()
    assert failed, f"mutant {name} passed every pin"
