"""The CPU oracle against closed forms, invariants, a worked example and brute
force (see tests/oracle_pins.py for what fixes each check)."""
import pytest

from tests import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    msg = check()
    assert msg is None, msg
