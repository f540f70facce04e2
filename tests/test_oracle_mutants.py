"""Plant plausible mistakes in copies of the oracle and show the pins catch each.

Every mutant is a text edit of ``oracle/attn_oracle.c`` compiled into a
temporary directory; the real oracle is untouched.  A mutant "survives" when
every pin in ``oracle_pins.ALL_CHECKS`` still passes, which would mean the pins
could not tell that mistake from the definition.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_CHECKS

MUTANTS = {
    "dropped_scale": [("s[j + 0] = scale * a0;", "s[j + 0] = a0;"),
                      ("s[j + 1] = scale * a1;", "s[j + 1] = a1;"),
                      ("s[j + 2] = scale * a2;", "s[j + 2] = a2;"),
                      ("s[j + 3] = scale * a3;", "s[j + 3] = a3;"),
                      ("s[j] = scale * a;", "s[j] = a;")],
    "causal_excludes_diagonal": [("n_vis = i + (Nk - Nq) + 1;", "n_vis = i + (Nk - Nq);")],
    "causal_top_left_alignment": [("n_vis = i + (Nk - Nq) + 1;", "n_vis = i + 1;")],
    "exp_sign_flipped": [("const double p = exp(s[j] - m) / l;", "const double p = exp(m - s[j]) / l;")],
    "lse_without_max": [("*lse_out = m + log(l);", "*lse_out = log(l);")],
    "sum_drops_first_key": [("for (j = 0; j < n_vis; ++j) l += exp(s[j] - m);",
                             "for (j = 1; j < n_vis; ++j) l += exp(s[j] - m);")],
    "v_transposed": [("o_row[d] += p * widen_bf16(vj[d]);", "o_row[d] += p * widen_bf16(vb[d * Nk + j]);")],
    "wrong_query_row": [("const uint16_t *qi = q + (bh * Nq + i) * D;",
                         "const uint16_t *qi = q + (bh * Nq + (Nq - 1 - i)) * D;")],
    "keys_of_head_zero": [("const uint16_t *kb = k + bh * Nk * D;", "const uint16_t *kb = k;")],
    "last_dim_dropped": [("for (d = 0; d < D; ++d) {\n            a0", "for (d = 0; d + 1 < D; ++d) {\n            a0")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for check in ALL_CHECKS:
        try:
            check(orc)
        except AssertionError as e:
            failures.append(check.__name__)
            if len(failures) >= 1:
                break
    assert failures, f"mutant {name} passed every pin"
