"""The oracle against its pins (CPU only): closed forms, numpy matmuls, invariants, brute
force and the hand-worked example.  See tests/oracle_pins.py for what each pin fixes."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_lib, check):
    check(oracle_lib)
