"""The CPU oracle against closed forms, library decoders, brute force and the pages'
stated properties (no GPU)."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_bucket_properties_exhaustive():
    fixed = pins.check_bucket_properties(65536)
    assert fixed[-1] == 65536
