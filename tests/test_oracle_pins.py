"""The oracle against its pins (see tests/oracle_checks.py for what pins what)."""
import pytest

import oracle
import oracle_checks as oc


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(lib, check):
    check(lib)
