"""Every planted mistake in the oracle must be caught by at least one pin.

Each case copies ``oracle/attn_oracle.c`` to a temporary directory, makes one
textual change that a plausible bug would make (a dropped term, a wrong sign,
a wrong index, a transposed operand, an off-by-one mask), compiles it, and
runs the pins against it.  The oracle itself is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("(p + 1 < nk ? p + 1 : nk)", "(p < nk ? p : nk)"),
    "no_max_shift": ("double w = exp(s[j] - m);", "double w = exp(s[j]);"),
    "sign_flip": ("double w = exp(s[j] - m);", "double w = exp(m - s[j]);"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "k_for_v": ("const double *vj = v + j * dv;", "const double *vj = k + j * d;"),
    "no_normalise": ("o[c] /= l;", "o[c] /= 1.0;"),
    "lse_drops_max": ("lse_rows[r] = m + log(l);", "lse_rows[r] = log(l);"),
    "key_index": ("const double *kj = k + j * d;", "const double *kj = k + j;"),
    "query_index": ("const double *q = q_rows + r * d;", "const double *q = q_rows + r;"),
    "max_not_updated": ("if (s[j] > m)\n                    m = s[j];", ""),
    "empty_policy": ("lse_rows[r] = -INFINITY;", "lse_rows[r] = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(path), str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
