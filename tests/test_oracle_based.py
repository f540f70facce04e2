"""The Based linear-attention oracle against facts fixed outside its own code,
and planted mistakes in copies of it that those facts must catch (no GPU)."""
import pytest

import oracle
from oracle_based_pins import ALL_BASED_CHECKS


@pytest.mark.parametrize("check", ALL_BASED_CHECKS, ids=[c.__name__ for c in ALL_BASED_CHECKS])
def test_based_oracle_pin(check):
    check(oracle.default())


# Each mutant is a text edit of oracle/based_oracle.c compiled on its own; the
# real oracle is untouched.
MUTANTS = {
    "no_quadratic_term": [("const double w = 1.0 + s + 0.5 * s * s;", "const double w = 1.0 + s;")],
    "quadratic_without_half": [("const double w = 1.0 + s + 0.5 * s * s;", "const double w = 1.0 + s + s * s;")],
    "linear_sign_flipped": [("const double w = 1.0 + s + 0.5 * s * s;", "const double w = 1.0 - s + 0.5 * s * s;")],
    "constant_dropped": [("const double w = 1.0 + s + 0.5 * s * s;", "const double w = s + 0.5 * s * s;")],
    "not_causal": [("for (j = 0; j <= i; ++j) {", "for (j = 0; j < N; ++j) {")],
    "diagonal_excluded": [("for (j = 0; j <= i; ++j) {", "for (j = 0; j < i || j == 0; ++j) {")],
    "not_normalised": [("for (d = 0; d < D; ++d) y_row[d] /= z;", "(void)z;")],
    "scale_dropped": [("const double s = scale * dot;", "const double s = dot;")],
    "value_of_query_row": [("const uint16_t *vj = vb + j * D;", "const uint16_t *vj = vb + i * D;")],
    "keys_of_head_zero": [("const uint16_t *kb = k + bh * N * F;", "const uint16_t *kb = k;")],
    "last_feature_dropped": [("for (a = 0; a < F; ++a) dot", "for (a = 0; a + 1 < F; ++a) dot")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_based_mutant_is_caught(name, tmp_path):
    with open(oracle.SOURCE_BASED) as f:
        src = f.read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    # The attention sources come along unchanged (the Oracle class binds them too).
    lib = oracle.compile_source([oracle.SOURCE, oracle.SOURCE_BWD, str(path)], str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    for check in ALL_BASED_CHECKS:
        try:
            check(orc)
        except (AssertionError, FloatingPointError, ZeroDivisionError):
            return
    pytest.fail(f"mutant {name} passed every pin")
