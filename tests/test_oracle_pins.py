"""The oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


def test_brute_force_helper_rejects_wrong_answers():
    # the brute-force reference itself: exactly one dominating subset
    import numpy as np
    vals = np.array([1.0, 1.0, 0.5])
    assert list(oracle_pins.brute_force_topk(vals, 1)) == [0]
    assert list(oracle_pins.brute_force_topk(vals, 2)) == [0, 1]
    assert not oracle_pins._dominates(vals, (1,))
