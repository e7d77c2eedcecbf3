"""Planted mistakes: the pins must catch plausible errors in the oracle.

Each case copies the oracle's C source, plants one mistake (a wrong tie rule,
a dropped sign, a transposed index, a wrong constant, ...), builds the copy on
the CPU and runs the pins against it.  A mistake that no pin notices fails
this test.  The oracle itself is never modified.
"""
import os
import subprocess

import pytest

import oracle
import test_gemm_oracle as gemm_pins
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.c")

# (name, original text, planted text)
MUTATIONS = [
    ("rn_tie_to_odd", "(dk == bestd && (k % 2) == 0)", "(dk == bestd && (k % 2) == 1)"),
    ("e4m3_overflow_to_nan", "if (v >= 448.0) return 0x7E;", "if (v >= 448.0) return 0x7F;"),
    ("e4m3_truncates", "double mant = rint(", "double mant = floor("),
    ("philox_wrong_key_word", "uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi1 ^ c1 ^ k1;"),
    ("philox_wrong_weyl", "k1 += W1;", "k1 += W0;"),
    ("philox_nine_rounds", "round < 10;", "round < 9;"),
    ("rht_not_normalised", "y[i] = (float)(0.25 * acc);", "y[i] = (float)(0.5 * acc);"),
    ("rht_signs_dropped", "double sj = ((signs >> j) & 1u) ? -1.0 : 1.0;", "double sj = 1.0;"),
    ("rht_transposed_index", "nvfp4ref_hadamard16(i, j) * sj", "nvfp4ref_hadamard16(i, (j + 1) & 15) * sj"),
    ("46_alpha_uses_448", "float denom = use46 ? 1536.0f : 2688.0f;", "float denom = use46 ? 2688.0f : 2688.0f;"),
    ("46_ties_pick_four", "if (s4 < s6) {", "if (s4 <= s6) {"),
    ("46_error_sign_flipped", "float err = fmaf(-val, d, z[i]);", "float err = fmaf(val, d, z[i]);"),
    ("mse_is_mae", "terms[i] = err * err;", "terms[i] = fabsf(err);"),
    ("tree_sequential", "float left = nvfp4ref_tree_sum(a, n / 2);\n  float right = nvfp4ref_tree_sum(a + n / 2, n / 2);\n  return left + right;",
     "float s = 0.0f;\n  for (int i = 0; i < n; ++i) s += a[i];\n  return s;"),
    ("sr_le_instead_of_lt", "return (u < p) ? hi : lo;", "return (u <= p) ? hi : lo;"),
    ("sr_col_uses_word0", "words[j] = w4[1]; /* columnwise copy: word 1 */", "words[j] = w4[0];"),
    ("sr_counter_transposed", "uint64_t i = counter_offset + (uint64_t)r * (uint64_t)N + (uint64_t)c;",
     "uint64_t i = counter_offset + (uint64_t)c * (uint64_t)N + (uint64_t)r;"),
    ("nibbles_swapped", "if (c % 2 == 0)\n    *p = (uint8_t)((*p & 0xF0) | (code & 0x0F));",
     "if (c % 2 == 1)\n    *p = (uint8_t)((*p & 0xF0) | (code & 0x0F));"),
    ("no_clamp_to_q", "float m = fminf(fabsf(v), (float)Q);", "float m = fabsf(v);"),
    ("sign_dropped", "codes[i] = (uint8_t)((sign << 3) | idx);", "codes[i] = (uint8_t)idx;"),
    ("scale_uses_q6_always", "float den = (float)Q * alpha;", "float den = 6.0f * alpha;"),
    ("gemm_b_uses_a_scales", "nvfp4ref_dequantize(qb, sb, alpha_b, N, K, 0, xb);",
     "nvfp4ref_dequantize(qb, sa, alpha_b, N, K, 0, xb);"),
    ("gemm_b_k_reversed", "acc += (double)xa[m * K + k] * (double)xb[n * K + k];",
     "acc += (double)xa[m * K + k] * (double)xb[n * K + (K - 1 - k)];"),
    ("gemm_drops_alpha_b", "nvfp4ref_dequantize(qb, sb, alpha_b, N, K, 0, xb);",
     "nvfp4ref_dequantize(qb, sb, 1.0f, N, K, 0, xb);"),
    ("gemm_float_accumulator", "double acc = 0.0;\n      for (int64_t k = 0; k < K; ++k) acc +=",
     "float acc = 0.0f;\n      for (int64_t k = 0; k < K; ++k) acc +="),
    ("2d_scale_not_replicated", "if (do_col) s_col[(tc + k) * (M / 16) + tr / 16] = e;", "if (do_col) s_col[(tc + k) * (M / 16) + tr / 16] = (uint8_t)(e + (k == 3));"),
]

# fast pins that take the oracle module as `ref`
PIN_FUNCS = [
    pins.test_grid_follows_printed_steps, pins.test_rn_ties_go_to_even_code,
    pins.test_e4m3_saturates_at_448, pins.test_four_is_two_thirds_of_block_max_at_scale_six,
    pins.test_value_at_75_percent_is_exact_three_at_scale_four,
    pins.test_tensor_scale_headroom_256_vs_448,
    pins.test_46_keeps_four_for_the_75_percent_block_and_six_for_an_exact_block,
    pins.test_tree_sum_is_adjacent_pairs_first, pins.test_hadamard_is_sylvester_and_orthogonal,
    pins.test_rht_preserves_norm_inner_products_and_inverts, pins.test_rht_signs_come_from_philox,
    pins.test_philox_known_answers, pins.test_sr_edge_cases, pins.test_zero_tensor,
    pins.test_2d_copies_are_transposes_and_dequantize_identically,
    pins.test_row_stripes_and_counter_offset_reproduce_the_whole,
    gemm_pins.test_gemm_equals_the_exact_rational_sum, gemm_pins.test_gemm_is_bilinear_in_scales_and_signs,
    gemm_pins.test_gemm_transpose_symmetry_and_reduction_order,
]
FLAG_SAMPLE = [1, 3, 3 | 64, 7, 3 | 16, 3 | 32, 3 | 16 | 32, 1 | 8 | 32 | 64, 7 | 32, 7 | 64]


def _caught(tmp_path, name, before, after, monkeypatch):
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not unique"
    mdir = tmp_path / name
    mdir.mkdir()
    (mdir / "nvfp4_oracle.c").write_text(src.replace(before, after))
    hdr = os.path.join(os.path.dirname(SRC), "nvfp4_oracle.h")
    (mdir / "nvfp4_oracle.h").write_text(open(hdr).read())
    so = mdir / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(mdir / "nvfp4_oracle.c"), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_LIB_PATH", str(so))
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    monkeypatch.setattr(oracle, "_lib", None)
    try:
        for f in PIN_FUNCS:
            try:
                f(oracle)
            except Exception:  # an assertion or any error counts as caught
                return f.__name__
        for flags in FLAG_SAMPLE:
            try:
                pins.test_oracle_matches_brute_force_on_tiny_tensors(oracle, flags)
            except Exception:  # an assertion or any error counts as caught
                return f"brute_force[{flags}]"
        return None
    finally:
        monkeypatch.setattr(oracle, "_lib", None)


@pytest.mark.parametrize("name,before,after", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, before, after):
    caught_by = _caught(tmp_path, name, before, after, monkeypatch)
    assert caught_by is not None, f"no pin caught the planted mistake {name}"
