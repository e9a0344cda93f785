"""The CPU oracle against its pins (brute force, closed forms, invariants).

Runs without a GPU. See tests/pins.py for what each pin checks and why.
"""
import pytest

from tests import pins


@pytest.fixture(scope="module")
def orc(oracle_mod):
    return oracle_mod.Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    import numpy as np

    q, k, v, ab, bb, ao, bo = pins.rng_inputs(1, 1, 4, 2, 1, 4)
    indptr, pos = pins.csr([[4]])  # position out of range
    with pytest.raises(ValueError):
        orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, 2, 1.0)
    indptr, pos = pins.csr([[1]])
    with pytest.raises(ValueError):
        orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, 0, 1.0)  # window < 1
    with pytest.raises(ValueError):
        orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, 2, 1.0, base_rows=np.array([5], np.int32))
