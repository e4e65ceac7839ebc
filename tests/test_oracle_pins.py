"""The oracle against its pins (closed forms, library softmax, brute force,
invariants, fault policy).  CPU only."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS,
                         ids=[c.__name__ for c in oracle_pins.ALL_CHECKS])
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)
