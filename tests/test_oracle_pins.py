"""The oracle against its pins (CPU only)."""
import pytest

from oracle_pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)
