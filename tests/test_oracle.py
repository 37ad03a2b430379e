"""The float64 oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    oracle.build()
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_streaming_lse_guards():
    """All -inf gives -inf; a block of only -inf carries no weight."""
    import math
    from oracle.online_model import streaming_lse
    assert streaming_lse([-math.inf] * 4) == -math.inf
    x = [-math.inf] * 7 + [0.5, 1.5] + [-math.inf] * 3
    assert abs(streaming_lse(x, block=7) - math.log(math.exp(0.5) + math.exp(1.5))) < 1e-15


def test_online_model_contract():
    """The block model raises on the pages' bad inputs (section "Check it")."""
    import numpy as np
    from oracle.online_model import online_attention
    bad = [((np.ones((4, 8)), np.ones((4, 7)), np.ones((4, 8))), ValueError),
           ((np.ones((4, 8)), np.ones((4, 8)), np.ones((5, 8))), ValueError),
           ((np.ones((2, 4, 8)), np.ones((4, 8)), np.ones((4, 8))), ValueError)]
    for args, err in bad:
        with pytest.raises(err):
            online_attention(*args)
