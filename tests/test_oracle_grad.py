"""The float64 gradient oracle against what mathematics fixes (CPU only)."""
import pytest

import oracle
import oracle_grad_pins


@pytest.fixture(scope="module")
def lib():
    oracle.build()
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_grad_pins.ALL_GRAD_PINS, ids=lambda p: p.__name__)
def test_grad_pin(lib, pin):
    pin(lib)


def test_grad_argument_errors(lib):
    import numpy as np
    with pytest.raises(ValueError):
        oracle.attention_grad(np.ones((4, 8)), np.ones((4, 7)), np.ones((4, 8)), np.ones((4, 8)))
    with pytest.raises(ValueError):
        oracle.attention_grad(np.ones((4, 8)), np.ones((4, 8)), np.ones((4, 8)), np.ones((3, 8)))
    # no keys: nothing to differentiate, all gradients zero
    dq, dk, dv = oracle.attention_grad(np.ones((3, 4)), np.ones((0, 4)), np.ones((0, 2)),
                                       np.ones((3, 2)))
    assert dq.shape == (3, 4) and dk.shape == (0, 4) and dv.shape == (0, 2)
    assert not dq.any()
