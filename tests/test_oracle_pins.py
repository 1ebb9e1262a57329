"""The fp64 oracle against facts fixed by the article's formulas and by mathematics."""
import pytest

import oracle
from _pins import ALL_PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)
