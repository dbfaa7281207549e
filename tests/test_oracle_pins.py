"""The CPU oracle against closed forms, invariants, brute force and the
textbook dense SwiGLU MLP (no GPU needed)."""
import pytest

import pin_checks


@pytest.mark.parametrize("check", pin_checks.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
