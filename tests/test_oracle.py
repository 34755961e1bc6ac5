"""The fp64 oracle against its pins (CPU only)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


def test_thread_count_does_not_change_results(orc):
    import numpy as np
    rng = np.random.default_rng(7)
    q, k, v, do = (rng.standard_normal((2, 37, 3, 16)) for _ in range(4))
    orc.set_threads(1)
    a = orc.attn_bwd(q, k, v, do, True)
    orc.set_threads(5)
    b = orc.attn_bwd(q, k, v, do, True)
    orc.set_threads(0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
