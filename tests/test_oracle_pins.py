"""The oracle against its pins, and each planted oracle mistake against them."""
import pytest

import oracle_pins
from oracle import oracle as orc


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(0)


# Each planted mistake (see OR_MUTATE in oracle/oracle.c) must fail a pin.
MUTATIONS = {
    1: "rope pairs interleaved",
    2: "rope sign flipped",
    3: "query misses its own key",
    4: "missing 1/sqrt(d)",
    5: "rmsnorm sum instead of mean",
    6: "silu without the factor z",
    7: "transposed weight operand",
    8: "first residual dropped",
    9: "gate and up swapped",
    10: "wrong in-block slot index",
    11: "mirror mode keeps n2 unrounded",
    12: "mirror mode keeps o unrounded",
}


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m].replace(" ", "_"))
def test_planted_mistake_is_caught(m):
    orc.build(m)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(m)
        except Exception:  # any disagreement or error counts as caught
            failed.append(pin.__name__)
    assert failed, f"mutation {m} ({MUTATIONS[m]}) passed every pin"
