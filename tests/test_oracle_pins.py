"""The oracle against its pins (closed forms, exact integers, brute force,
invariants and the pages' worked examples).  CPU only."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_tolerance_formula():
    # 1e-5 * sum|x| + 1e-6, per output element.
    assert oracle.tolerance(0.0) == pytest.approx(1e-6, rel=0, abs=1e-18)
    assert oracle.tolerance(1e5) == pytest.approx(1.000001, rel=1e-15)
