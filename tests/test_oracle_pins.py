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


def test_memory_table_golden_is_consistent():
    """CS336 L5 section 8.5's table, checked as arithmetic on the printed
    figures (not an oracle pin: no oracle result is involved).  The extra
    memory FlashAttention keeps is one fp32 logsumexp per query row, against
    two n x n bf16 matrices (S and P) for the standard implementation."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "cs336_l5_memory_table.json")
    with open(path) as f:
        g = json.load(f)
    for row in g["rows"]:
        n = row["n"]
        assert round(n * 4 / 1e6, 2) == row["flash_extra_MB"], n
        digits = 1 if row["standard_GB"] >= 10 else 2
        assert round(2 * n * n * 2 / 1e9, digits) == row["standard_GB"], n
