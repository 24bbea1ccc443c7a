"""The fp64 oracle against values the pages print and facts the mathematics
fixes (no GPU needed)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(oracle)


def test_oracle_rejects_causal_with_more_queries_than_keys():
    """Causal attention of Nq > Nk queries would leave the first Nq - Nk rows
    with no visible key; the oracle refuses it, as the library does."""
    import numpy as np
    import oracle
    q, k = np.zeros((1, 1, 5, 4)), np.zeros((1, 1, 3, 4))
    for fn in (oracle.attention, oracle.attention_blocked):
        with pytest.raises(ValueError):
            fn(q, k, k, causal=True)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, k, k, [[0, 0]], causal=True)
    o, _ = oracle.attention(q, k, k, causal=False)  # non-causal is defined
    assert o.shape == (1, 1, 5, 4)
