"""The oracle against its pins (CPU only): see ``oracle_pins``."""
from __future__ import annotations

import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    check(orc)


def test_worked_examples_cover_every_reading():
    """The fixture holds an example for each reading it is meant to pin."""
    names = {n for n, *_ in oracle_pins.load_worked_examples()}
    for needed in ("order_tie_then_cancel", "fp32_accumulation", "tie_to_even_down",
                   "tie_to_even_up", "all_negative_zero", "eight_copies_exact",
                   "single_rank_identity", "subnormal_sum", "bf16_overflow_tie"):
        assert needed in names
