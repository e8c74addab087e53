"""The pins catch plausible mistakes: each test here plants one mistake in a
copy of the oracle's C source (on the CPU, in a temporary directory), compiles
it, swaps it in for the real oracle and checks that at least one pin fails."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTATIONS = {
    "kv_head_modulo": ("const int kvh = h / g;", "const int kvh = h % Hkv;"),
    "dropped_scale": ("s[t - start] = scale * dot;", "s[t - start] = dot;"),
    "wrong_slot": ("+ (t % page_size)) * D;\n            for (int d = 0; d < D; ++d) kd[d]",
                   "+ ((t + 1) % page_size)) * D;\n            for (int d = 0; d < D; ++d) kd[d]"),
    "f32_as_bf16": ("if (dtype == 2) return (double)((const float*)base)[e];",
                    "if (dtype == 2) return bf16_bits_to_double(((const uint16_t*)base)[e]);"),
    "window_off_by_one": ("const int start = (window > 0 && window < L) ? L - window : 0;\n"
                          "        const int n",
                          "const int start = (window > 0 && window < L) ? L - window + 1 : 0;\n"
                          "        const int n"),
    "base2_lse": ("const double l = M + log(Z);", "const double l = M + log2(Z);"),
    "unnormalised_weights": ("const double w = exp(s[t - start] - l);",
                             "const double w = exp(s[t - start] - M);"),
    "k_in_place_of_v": ("o[d] += w * elem(v_cache, vrow + d, dtype);",
                        "o[d] += w * elem(k_cache, vrow + d, dtype);"),
    "half_exponent_bias": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "bf16_exponent_bias": ("ldexp((double)(128 + m), e - 134)", "ldexp((double)(128 + m), e - 133)"),
    "rope_sign": ("x[i] = a * c - b * sn;", "x[i] = a * c + b * sn;"),
    "rope_query_position": ("rope_rotate(qd, D, rope_theta, (double)(L - 1));\n\n",
                            "rope_rotate(qd, D, rope_theta, (double)L);\n\n"),
    "rope_frequency": ("pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)"),
}


def _checks():
    yield lambda: pins.test_matches_dense_textbook_attention(*pins.SMALL[4])
    yield lambda: pins.test_matches_dense_textbook_attention(*pins.SMALL[2])
    yield pins.test_closed_form_golden_cases
    yield lambda: pins.test_window_equals_truncated_context(17)
    yield lambda: pins.test_bf16_inputs_match_dense_textbook_attention(*pins.SMALL[2])
    yield lambda: pins.test_rope_matches_complex_rotation_reference(64, 10000.0)
    yield lambda: pins.test_fp32_inputs_match_dense_textbook_attention(*pins.SMALL[2])


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmut.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(mutated), "-o",
                    lib_path, "-lm"], check=True, capture_output=True)
    saved = oracle._lib
    oracle._lib = oracle.bind(lib_path)
    failed = 0
    try:
        for check in _checks():
            try:
                check()
            except (AssertionError, oracle.OracleError):
                failed += 1
    finally:
        oracle._lib = saved
    assert failed > 0, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_the_same_checks():
    for check in _checks():
        check()
    assert np.isfinite(oracle.half_to_double(0x3C00))
