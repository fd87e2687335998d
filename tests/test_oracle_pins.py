"""The CPU oracle against facts outside itself (see tests/oracle_pins.py for what pins what)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.default())


def test_oracle_rejects_bad_shapes():
    import numpy as np

    o = oracle.default()
    rng = np.random.default_rng(0)
    p = oracle_pins.random_params(rng, 1, 2, 4)
    with pytest.raises(ValueError):
        o.forward(np.zeros((1, 1, 6, 8)), p)  # even k
