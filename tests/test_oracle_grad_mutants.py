"""Every planted mistake in the gradient oracle must be caught by a pin.

Each case copies ``oracle/attn_grad_oracle.c`` to a temporary directory,
makes one textual change that a plausible bug would make, compiles it with
the unchanged forward oracle, and runs the gradient pins against it.
"""
import os

import pytest

import oracle
import oracle_grad_pins

HERE = os.path.dirname(oracle.__file__)
SRC = os.path.join(HERE, "attn_grad_oracle.c")
FWD = os.path.join(HERE, "attn_oracle.c")

MUTANTS = {
    "no_delta_in_dq": ("const double ds = s[j] * (dp - delta);", "const double ds = s[j] * dp;"),
    "no_delta_in_dk": ("const double ds = p * (dp - delta[i]);", "const double ds = p * dp;"),
    "dq_without_scale": ("dq[c] += scale * ds * kj[c];", "dq[c] += ds * kj[c];"),
    "dk_without_scale": ("dk[c] += scale * ds * qi[c];", "dk[c] += ds * qi[c];"),
    "dq_uses_values": ("const double *kj = k + j * d;\n                for", "const double *kj = v + j * dv;\n                for"),
    "dv_uses_ds": ("dvr[c] += p * g[c];", "dvr[c] += ds * g[c];"),
    "delta_from_values": ("delta += g[c] * o[c];", "delta += g[c] * v[c];"),
    "key_pass_causal_off_by_one": ("const int64_t first = causal ? (k_pos[r] < 0 ? 0 : k_pos[r]) : 0;",
                                   "const int64_t first = causal ? (k_pos[r] < 0 ? 0 : k_pos[r] + 1) : 0;"),
    "query_pass_causal_off_by_one": ("return pos + 1 < nk ? pos + 1 : nk;", "return pos < nk ? pos : nk;"),
    "p_without_lse": ("const double p = exp(scale * dot - lse[i]);", "const double p = exp(scale * dot);"),
    "lse_without_max": ("const double lse = m + log(l);", "const double lse = log(l);"),
    "dk_sign": ("dk[c] += scale * ds * qi[c];", "dk[c] -= scale * ds * qi[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_grad_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant_grad.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_oracle([FWD, str(path)], str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    caught = []
    for pin in oracle_grad_pins.ALL_GRAD_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
