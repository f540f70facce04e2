"""The backward oracle against facts fixed outside its own code, and planted mistakes."""
import pytest

import oracle
from oracle_bwd_pins import ALL_BWD_CHECKS


@pytest.mark.parametrize("check", ALL_BWD_CHECKS, ids=[c.__name__ for c in ALL_BWD_CHECKS])
def test_bwd_oracle_pin(check):
    check(oracle.default())


MUTANTS = {
    "dq_without_scale": [("dqi[d] += scale * ds * k[j * D + d];", "dqi[d] += ds * k[j * D + d];")],
    "dk_uses_k": [("dk[j * D + d] += scale * ds * qi[d];", "dk[j * D + d] += scale * ds * k[j * D + d];")],
    "dv_without_p": [("dv[j * D + d] += p[j] * doi[d];", "dv[j * D + d] += doi[d];")],
    "delta_dropped": [("const double ds = p[j] * (dp[j] - dl);", "const double ds = p[j] * dp[j];")],
    "dp_uses_k": [("for (d = 0; d < D; ++d) a += doi[d] * v[j * D + d];", "for (d = 0; d < D; ++d) a += doi[d] * k[j * D + d];")],
    "ds_sign": [("const double ds = p[j] * (dp[j] - dl);", "const double ds = p[j] * (dl - dp[j]);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE_BWD).read()
    for old, new in MUTANTS[name]:
        assert old in src, old
        src = src.replace(old, new)
    path = tmp_path / "bwd_mutant.c"
    path.write_text(src)
    orc = oracle.Oracle(oracle.compile_source([oracle.SOURCE, str(path)], str(tmp_path / "libmut.so")))
    caught = False
    for check in ALL_BWD_CHECKS:
        try:
            check(orc)
        except AssertionError:
            caught = True
            break
    assert caught, f"backward mutant {name} passed every pin"
