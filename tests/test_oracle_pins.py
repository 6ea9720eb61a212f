"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import _pins


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    check(orc)
