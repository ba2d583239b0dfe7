"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle_pins as P  # noqa: E402


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
