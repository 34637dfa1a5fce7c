"""The oracle pinned to things other than itself (see tests/oracle_checks.py)."""
import pytest

import oracle_checks as C


@pytest.mark.parametrize("check", C.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)
