"""The oracle against its pins (CPU only), and each planted mistake against the pins."""
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


# Each build plants one plausible mistake in the oracle (see the PLANT notes in
# pa_oracle.c): 1 scale dropped, 2 interleaved head groups, 3 causal limit off
# by one, 4 offsets reversed inside a block, 5 a softmax term left out of the
# denominator, 6 chunk rows reversed, 7 V read from the K cache, 8 the speculative
# acceptance ratio inverted, 9 the speculative residual taken the wrong way round, 10 the E4M3
# exponent bias off by one, 11 E4M3 encoding truncating instead of rounding to nearest even, 12
# copy-on-write block copies made the wrong way, 13 the K and V dequantisation scales swapped,
# 14 the append's block and in-block offset swapped.
@pytest.mark.parametrize("plant", list(range(1, 15)))
def test_planted_mistake_is_caught(plant):
    bad = oracle.load(plant)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} slipped past every pin"
