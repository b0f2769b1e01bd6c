"""The fp64 oracle against its pins (CPU only; see oracle_pins.py)."""
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_oracle_uses_threads(lib):
    assert oracle.num_threads(lib) >= 1


def test_oracle_rejects_out_of_range_slot(lib):
    import numpy as np
    q = np.zeros((1, 1, 8), np.uint16)
    kv = np.zeros((4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.sda_decode(q, kv, [4], [0, 1], [0.0], 1.0, lib=lib)
    with pytest.raises(ValueError):
        oracle.sda_decode(q, kv, [0, 1], [1, 0], [0.0], 1.0, lib=lib)
