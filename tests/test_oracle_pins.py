"""The CPU oracle against its pins, and the pins against planted mistakes.

The pins themselves are in tests/pins.py; each rests on something other than
the oracle (hand-derived bytes and worked examples, big-integer and numpy
library routines, brute force, closed forms, the quantiser invariant).
"""
import tempfile
from pathlib import Path

import pytest

import oracle
from pins import PINS


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(o, pin):
    pin(o)


# Each planted mistake is a plausible error in reading the pages: the old
# num_groups x N scale layout, a zero point instead of an additive zero, MSB-first
# bits, a wrong group index, a dropped term, a transposed operand, a wrong fp16
# exponent bias, the sign of the exponent in silu, gate and up swapped; in the
# quantiser, ties rounded half away from zero, the last (not the first) of equal
# minima, and a constant group's scale left at 2^-14.
PLANTS = ["PLANT_STREAM_MSB", "PLANT_CODE_MSB", "PLANT_GROUP_MOD", "PLANT_SZ_TRANSPOSED",
          "PLANT_DROP_ZERO", "PLANT_ZERO_POINT", "PLANT_DROP_BIAS", "PLANT_X_TRANSPOSED",
          "PLANT_HALF_BIAS", "PLANT_LAST_K", "PLANT_SILU_SIGN", "PLANT_SILU_SWAP",
          "PLANT_ROUND_HALF_AWAY", "PLANT_MIN_LAST", "PLANT_CONST_SCALE_FLOOR"]


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_fails_a_pin(plant):
    with tempfile.TemporaryDirectory() as d:
        lib = oracle.build(defines=(plant,), out=Path(d) / f"lib_{plant}.so")
        bad = oracle.Oracle(oracle.load(lib))
        failed = []
        for pin in PINS:
            try:
                pin(bad)
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"{plant} passed every pin"
