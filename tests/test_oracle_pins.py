"""The fp64 oracle against its pins (library decoders, torch SDPA, closed forms,
invariances and the pages' worked examples)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())
