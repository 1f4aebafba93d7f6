"""The CPU oracle against its pins (see ``oracle_pins.py``), and the pins
against oracle builds with planted mistakes."""

import pytest

from oracle import Oracle
from oracle_pins import MUTANTS, PINS


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(oracle, name):
    ok, detail = PINS[name](oracle)
    assert ok, detail


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistake(mutant):
    o = Oracle(mutant)
    assert o.lib.oracle_mutant() == mutant
    failed = []
    for name, pin in PINS.items():
        try:
            ok, _ = pin(o)
        except Exception:
            ok = False
        if not ok:
            failed.append(name)
    assert failed, f"planted mistake {mutant} passed every pin"


def test_fp32_form_thread_split_is_exact():
    """Splitting rows over threads must not change any result."""
    import numpy as np
    import synth
    inp = synth.make_inputs(37, 512, 3, 4, 64, 9)
    o = Oracle(0)
    w = o.pack(inp.q, 4)
    y1, _, used1 = o.qmv_f32_factored(w, inp.scales, inp.biases, inp.x, 4, 64, nthreads=1)
    y4, _, used4 = o.qmv_f32_factored(w, inp.scales, inp.biases, inp.x, 4, 64, nthreads=4)
    assert used1 == 1 and used4 == 4
    assert np.array_equal(y1, y4)
