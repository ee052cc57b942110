"""The oracle against values and properties fixed by the pages and by mathematics."""
import pytest

import oracle_pins
from oracle import awq_oracle


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(awq_oracle)


def test_alpha_grid_is_twenty_steps():
    g = awq_oracle.alpha_grid(21)
    assert g[0] == 0.0 and g[-1] == 1.0 and len(g) == 21
    assert abs(g[1] - 0.05) < 1e-15 and abs(g[10] - 0.5) < 1e-15


def test_nonfinite_and_overflow_are_errors():
    import numpy as np
    X = np.ones((4, 8), dtype=np.float32)
    X[1, 2] = np.nan
    with pytest.raises(awq_oracle.OracleNonFiniteError):
        awq_oracle.act_stats(X)
    W = np.full((8, 2), 1e6, dtype=np.float32)
    with pytest.raises(awq_oracle.OracleRangeError):
        awq_oracle.quantize_groups(W, 8, True)


def test_degenerate_zero_group():
    import numpy as np
    W = np.zeros((16, 3), dtype=np.float32)
    for sym in (False, True):
        codes, step, zero = awq_oracle.quantize_groups(W, 8, sym)
        assert np.all(step == 0)
        deq = awq_oracle.dequantize(codes, step, zero, 8)
        assert np.all(deq == 0)
