"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

from pins import ALL_CHECKS, exhaustive_bf16_rounding


@pytest.mark.parametrize("check", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_oracle_pin(check):
    check()


def test_bf16_rounding_on_every_fp32_bit_pattern():
    exhaustive_bf16_rounding()
