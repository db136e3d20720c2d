"""The CPU oracle against its pins (fixtures, closed forms, invariants,
library routines on special cases, brute force on tiny inputs)."""
from __future__ import annotations

import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_group(orc):
    import numpy as np
    with pytest.raises(ValueError):
        orc.quantize(np.zeros((2, 200), dtype=np.uint16), 128)
