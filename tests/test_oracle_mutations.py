"""Plant one plausible slip at a time in a copy of the C oracle and check that
the pin suite rejects every mutant.  Runs on the CPU only; the mutants are
built into a temporary directory and never touch the real oracle."""

import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")

# (name, exact text in fa_oracle.c, replacement).  Every mutant stays in bounds.
MUTATIONS = [
    ("dropped_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("exp_sign", "s[j] = exp(s[j] - M);", "s[j] = exp(M - s[j]);"),
    ("max_not_subtracted", "s[j] = exp(s[j] - M);", "s[j] = exp(s[j]);"),
    ("mask_hides_diagonal", "if (causal && j > pos) {", "if (causal && j >= pos) {"),
    ("mask_leaks_next_key", "if (causal && j > pos) {", "if (causal && j > pos + 1) {"),
    ("offset_ignored_forward",
     "score_row(q_head + i * d, k_head, Nk, d, scale, causal, i + q_offset, P + r * Nk);",
     "score_row(q_head + i * d, k_head, Nk, d, scale, causal, i, P + r * Nk);"),
    ("no_normalisation", "for (int64_t j = 0; j < Nk; ++j) s[j] /= Z;", ""),
    ("lse_without_max", "M + log(Z);", "log(Z);"),
    ("pv_uses_keys",
     "const double* v_row = v_head + j * d;\n        for (int64_t c = 0; c < d; ++c) o_row[c]",
     "const double* v_row = k_head + j * d;\n        for (int64_t c = 0; c < d; ++c) o_row[c]"),
    ("gqa_modulo_mapping", "h = u % Hq, hk = h / G;", "h = u % Hq, hk = h % Hkv;"),
    ("bwd_group_strided", "const int64_t h = hk * G + g;", "const int64_t h = g * Hkv + hk;"),
    ("bwd_jacobian_sign", "(dP[i * Nk + j] - r)", "(dP[i * Nk + j] + r)"),
    ("bwd_dq_unscaled", "for (int64_t c = 0; c < d; ++c) dq_row[c] *= scale;", ""),
    ("bwd_dk_unscaled", "dk_row[c] += scale * ds * q_row[c];", "dk_row[c] += ds * q_row[c];"),
    ("bwd_dv_from_ds", "const double p = P[i * Nk + j];\n          if (p == 0.0) continue;\n"
                       "          double* dv_row",
     "const double p = dP[i * Nk + j];\n          if (p == 0.0) continue;\n"
     "          double* dv_row"),
    ("bwd_dp_uses_keys",
     "const double* v_row = v_head + j * d;\n          double acc = 0.0;",
     "const double* v_row = k_head + j * d;\n          double acc = 0.0;"),
    ("row_dot_wrong_operand", "acc += a[r * d + c] * b[r * d + c];",
     "acc += a[r * d + c] * a[r * d + c];"),
    ("bwd_dq_uses_values",
     "const double* k_row = k_head + j * d;\n          for (int64_t c = 0; c < d; ++c) dq_row",
     "const double* k_row = v_head + j * d;\n          for (int64_t c = 0; c < d; ++c) dq_row"),
]


def _caught(orc):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle"
    mutant = tmp_path / f"{name}.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.build(str(mutant), str(tmp_path / f"lib{name}.so"))
    failed = _caught(oracle.load(lib))
    assert failed, f"no pin caught mutant {name}"
