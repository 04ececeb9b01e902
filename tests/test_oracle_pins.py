"""The CPU oracle against what the pages and the mathematics fix (no GPU needed)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=[c.__name__ for c in P.ALL_CHECKS])
def test_oracle_pin(check):
    ok, msg = check()
    assert ok, msg
