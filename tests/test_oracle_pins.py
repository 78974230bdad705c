"""The CPU oracle against its pins (no GPU).  See tests/oracle_pins.py."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)
