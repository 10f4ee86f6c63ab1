"""The fp64 oracle against its pins: closed forms, invariants, brute force."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.library())


def test_every_operator_is_pinned():
    names = [p.__name__ for p in oracle_pins.ALL_PINS]
    assert sum(n.startswith("pin_layernorm_") for n in names) >= 4
    for op in ("softmax", "rmsnorm", "xent"):
        assert sum(n.startswith(f"pin_{op}_") and "_bwd_" not in n for n in names) >= 5, op
        assert sum(n.startswith(f"pin_{op}_bwd_") for n in names) >= 3, op
