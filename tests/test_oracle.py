"""Pins of the fp64 oracle (CPU only): every check in oracle_pins must hold."""
import pytest

from oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check()
