"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a private copy of the oracle's C source,
compiles it into a temporary library, points the oracle front end at it and
runs the pins of test_oracle_pins.py. At least one pin must fail for every
mutant; the real oracle passes all of them (test_oracle_pins.py itself).
"""
import os
import subprocess

import pytest

from oracle import causal_gqa as orc
from tests import test_oracle_pins as pins
from tests import test_oracle_prep_pins as prep_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "causal_gqa_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("drops the diagonal key", "const int64_t n_causal = i - s_b + 1;",
     "const int64_t n_causal = i - s_b + (i > s_b ? 0 : 1);"),
    ("sees one future key", "const int64_t n_causal = i - s_b + 1;",
     "const int64_t n_causal = i - s_b + 1 + (i + 1 < cu[b + 1] ? 1 : 0);"),
    ("bidirectional rows stop at the query", "const int64_t n = causal ? n_causal : e_b - s_b;",
     "const int64_t n = causal ? n_causal : n_causal;"),
    ("wrong GQA head (modulo)", "const int g = (int)(((int64_t)h * hkv) / hq);",
     "const int g = h % hkv;"),
    ("scale not applied", "z[jj] = scale * dot;", "z[jj] = dot;"),
    ("max not added back to the LSE", "const double L = m + log(sum);",
     "const double L = log(sum) + (m > 0 ? 0.0 : m);"),
    ("values read from k", "const uint16_t *vrow = v + ", "const uint16_t *vrow = k + "),
    ("keys taken from the tensor start, not the sequence start",
     "k + ((int64_t)g * T + s_b + jj) * d", "k + ((int64_t)g * T + jj) * d"),
    ("query read from the KV head", "q[((int64_t)h * T + i) * d + c]",
     "q[((int64_t)g * T + i) * d + c]"),
    ("probabilities not normalised", "const double p = exp(z[jj] - L);",
     "const double p = exp(z[jj] - m);"),
]

PREP_MUTANTS = [
    ("rotation pairs neighbours", "const double a = y[i], b = y[i + half];",
     "const double a = y[i], b = y[(i + 1) % d];"),
    ("rotation sign", "y[i] = a * cs - b * sn;", "y[i] = a * cs + b * sn;"),
    ("norm weight dropped", "y[c] = y[c] * inv * bf16_bits_to_double(w[c]);",
     "y[c] = y[c] * inv;"),
    ("sum instead of mean", "ms /= d;", "ms /= 1;"),
    ("eps dropped", "const double inv = 1.0 / sqrt(ms + eps);", "const double inv = 1.0 / sqrt(ms);"),
]

PIN_CALLS = [
    ("bruteforce-0", lambda: pins.test_oracle_matches_dense_bruteforce(*pins.SHAPES[2])),
    ("bruteforce-varlen", lambda: pins.test_oracle_matches_dense_bruteforce(*pins.SHAPES[4])),
    ("sdpa", lambda: pins.test_oracle_matches_torch_sdpa_float64((9, 23), 4, 2, 32)),
    ("first-row", pins.test_first_row_closed_form),
    ("zero-scale", pins.test_zero_scale_gives_prefix_mean),
    ("one-hot", pins.test_one_hot_logit_selects_its_value_row),
    ("constant-v", pins.test_constant_v_gives_constant_output),
    ("probs", pins.test_probability_rows_sum_to_one_and_are_causal),
    ("future", pins.test_future_keys_do_not_matter),
    ("gqa-repeat", pins.test_gqa_equals_explicit_kv_repetition),
    ("varlen", pins.test_varlen_equals_separate_calls),
    ("key-shift", pins.test_common_key_shift),
    ("bidir-brute", lambda: pins.test_bidirectional_matches_dense_bruteforce((17,), 2, 1, 8)),
    ("bidir-sdpa", pins.test_bidirectional_matches_torch_sdpa_float64),
    ("bidir-perm", pins.test_bidirectional_is_invariant_to_key_order),
    ("bidir-zero", pins.test_bidirectional_zero_scale_and_last_row),
]


def _build_mutant(tmp_path, name, old, new):
    with open(SRC) as fh:
        src = fh.read()
    assert src.count(old) == 1, "mutation site not found once: %r" % old
    path_c = tmp_path / "mutant.c"
    path_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o",
                    str(lib), str(path_c), "-lm"], check=True)
    return str(lib)


PREP_PIN_CALLS = [
    ("rms-torch", prep_pins.test_rms_norm_matches_torch_float64),
    ("unit-ms", prep_pins.test_unit_weight_gives_unit_mean_square_and_eps_shift),
    ("scale-inv", prep_pins.test_norm_is_scale_invariant),
    ("identity", prep_pins.test_identity_tables_leave_rows_unchanged),
    ("pair-norms", prep_pins.test_rotation_keeps_pair_norms),
    ("relative", prep_pins.test_rotated_dot_product_depends_on_position_difference),
    ("angles-add", prep_pins.test_rotation_angles_add),
]


@pytest.mark.parametrize("name,old,new", PREP_MUTANTS, ids=[m[0] for m in PREP_MUTANTS])
def test_prep_pins_catch_mutant(tmp_path, monkeypatch, name, old, new):
    lib = orc.bind(_build_mutant(tmp_path, name, old, new))
    monkeypatch.setattr(orc, "_LIB", lib)
    caught = []
    for pin_name, call in PREP_PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin_name)
    assert caught, "no pin caught the planted mistake: %s" % name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, monkeypatch, name, old, new):
    lib = orc.bind(_build_mutant(tmp_path, name, old, new))
    monkeypatch.setattr(orc, "_LIB", lib)
    caught = []
    for pin_name, call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin_name)
    assert caught, "no pin caught the planted mistake: %s" % name
