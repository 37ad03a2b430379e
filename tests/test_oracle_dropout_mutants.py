"""Every planted mistake in the dropout oracle must be caught by a pin.

Each case copies ``oracle/attn_dropout_oracle.c`` to a temporary directory,
makes one textual change that a plausible bug would make, compiles it with
the unchanged forward and gradient oracles, and runs the dropout pins
against it.
"""
import os

import pytest

import oracle
import oracle_dropout_pins

HERE = os.path.dirname(oracle.__file__)
SRC = os.path.join(HERE, "attn_dropout_oracle.c")
OTHERS = [os.path.join(HERE, "attn_oracle.c"), os.path.join(HERE, "attn_grad_oracle.c")]

MUTANTS = {
    "philox_multiplier": ("const uint32_t M0 = 0xD2511F53u", "const uint32_t M0 = 0xD2511F55u"),
    "philox_no_key_bump": ("            k1 += W1;\n", ""),
    "philox_nine_rounds": ("for (int r = 0; r < 10; ++r)", "for (int r = 0; r < 9; ++r)"),
    "keep_at_threshold": ("return byte < (uint32_t)t;", "return byte <= (uint32_t)t;"),
    "output_not_rescaled": ("oi[c] *= s / l;", "oi[c] *= 1.0 / l;"),
    "normaliser_of_kept_weights": ("        l += e;\n", "        l += keep(bh, i, j, seed, offset, t) ? e : 0.0;\n"),
    "dp_without_mask": ("dp[j] = z ? s * gv : 0.0;", "dp[j] = s * gv;"),
    "dv_without_scale": ("dvv[j * dv + c] += s * pr[j] * gi[c];", "dvv[j * dv + c] += pr[j] * gi[c];"),
    "offset_ignored": ("const int64_t last = i + 1 + q_off;", "const int64_t last = i + 1;"),
    "mask_by_position": ("            if (keep(bh, i, j, seed, offset, t))",
                         "            if (keep(bh, i + q_off, j, seed, offset, t))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_dropout_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant_dropout.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_oracle(OTHERS + [str(path)], str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    caught = []
    for pin in oracle_dropout_pins.ALL_DROPOUT_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
