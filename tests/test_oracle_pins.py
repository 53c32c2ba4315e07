"""The fp64 oracle pinned to what the pages and mathematics fix (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    msg = check()
    assert msg is None, msg


def test_oracle_reports_threads():
    import oracle
    assert oracle.num_threads() >= 1
