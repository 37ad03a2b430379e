"""Pins of the float64 dropout oracle (CPU only).

The pages say only that, with dropout, the generator's state is kept so the
backward pass regenerates the same mask ("Why FlashAttention Can Avoid a
Square Attention Array Without Making Attention Linear", section "Backward
can recreate tiles instead of retaining the square").  The oracle's
generator, keep rule and gradients are pinned here against things outside
its own code: the generator's published known-answer vectors, the exact
reduction to the dropout-free oracle at p = 0, the keep rate's binomial
law, the unbiasedness the 256 / t scale is there for, and finite
differences of the loss with the mask held fixed.
"""
import pytest

import oracle
import oracle_dropout_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_DROPOUT_PINS, ids=lambda f: f.__name__)
def test_dropout_pin(pin):
    pin(oracle.load())


def test_threshold_reading():
    """t = floor((1 - p) * 256 + 1/2): halves round up (not to even)."""
    assert oracle.dropout_threshold(1 - 128.5 / 256) == 129
    assert oracle.dropout_threshold(0.0) == 256
    assert oracle.dropout_threshold(0.1) == 230
    assert oracle.dropout_threshold(0.5) == 128
    for bad in (1.0, -0.1, 0.999):
        with pytest.raises(ValueError):
            oracle.dropout_threshold(bad)
