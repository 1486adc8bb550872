"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__[4:])
def test_pin(o, pin):
    pin(o)


def test_threads_do_not_change_results(o):
    import numpy as np
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 8, 32)).astype(np.float32)
    K = rng.standard_normal((2, 2, 100, 32)).astype(np.float32)
    V = rng.standard_normal((2, 2, 100, 32)).astype(np.float32)
    a, la = o.decode(q, K, V, [100, 57], 0.2, threads=1)
    b, lb = o.decode(q, K, V, [100, 57], 0.2, threads=4)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
