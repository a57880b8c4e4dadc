"""The FP64 oracle against closed forms, invariants, finite differences and
torch's own cross_entropy (CPU only)."""
import pytest

import oracle.lce_oracle as orc
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    assert pin(orc) == []


def test_label_range_is_an_error():
    import numpy as np
    X, W, b, y = oracle_pins.tiny_problem(0)
    y[0] = W.shape[0]
    with pytest.raises(ValueError):
        orc.forward(X, W, b, y)
    y[0] = -1
    with pytest.raises(ValueError):
        orc.forward(X, W, b, y)
    y[0] = -100
    orc.forward(X, W, b, y)
    assert np.isfinite(orc.forward(X, W, b, y)["loss"])
