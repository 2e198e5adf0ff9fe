"""The CPU oracle against mathematics and library routines (no GPU)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod.default())


def test_golden_fixtures_reproduce(oracle_mod):
    """The oracle still writes the stored fixtures bit for bit."""
    from tests import golden
    for name in golden.FIXTURES:
        g = golden.load(name)
        if "X" in g:
            got = oracle_mod.ffn_gated(g["X"], g["W1"], g["W3"])
        else:
            act = "gelu_tanh" if "gelu" in name else ("silu" if "silu" in name else "none")
            got = oracle_mod.linear(g["A"], g["B"], bias=g.get("bias"), R=g.get("R"), act=act)
        assert (got == g["D"]).all(), name
