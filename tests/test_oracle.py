"""The CPU oracle against its pins (no GPU). See tests/oracle_pins.py for the facts used."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(o, check):
    check(o)
