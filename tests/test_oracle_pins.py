"""The oracle checked against the pages, the format specifications and the
mathematics (see tests/pins.py for the independent route each pin takes)."""
import pytest

import oracle as O
import pins


@pytest.fixture(scope="module")
def lib():
    return O.load()


@pytest.mark.parametrize("pin", pins.FAST_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("fmt", pins.INT_FORMATS)
@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("absmax", [1.2265625, 0.0078125, 3.0])
def test_rounding_exhaustive(lib, fmt, src, absmax):
    """Every finite 16-bit input at or below the block absmax, for every width."""
    pins.pin_rounding_exhaustive_16bit(lib, fmt=fmt, src=src, absmax=absmax)
