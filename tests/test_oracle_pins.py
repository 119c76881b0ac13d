"""The fp64 oracle against facts it does not produce itself (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, oracle_mod):
    check(oracle_mod.default())
