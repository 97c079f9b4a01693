"""The CPU oracle against facts outside itself (formats, closed forms, exact
arithmetic).  CPU only."""
import pytest

import oracle

from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_golden_fixture_replays():
    """The oracle built on this machine reproduces the stored fixture bits
    (written by tests/golden/make_golden.py from the oracle alone)."""
    import numpy as np

    from golden_io import cases

    n = 0
    for c in cases():
        d, dt, eps = c["inputs"], c["dtype"], c["eps"]
        if c["op"] == "rms_norm":
            r = oracle.rms_norm(d["x"], d["gamma"], eps, dt)
        elif c["op"] == "fused_add_rms_norm":
            r = oracle.fused_add_rms_norm(d["x"], d["residual"], d["gamma"], eps, dt)
        else:
            r = oracle.reduce_add_rms_norm(d["partials"], d["residual"], d["gamma"], eps, dt)
        assert np.array_equal(r.y.view(np.uint8), c["expected"]["y"].view(np.uint8)), c["op"]
        if "residual" in c["expected"]:
            assert np.array_equal(r.residual.view(np.uint8),
                                  c["expected"]["residual"].view(np.uint8)), c["op"]
        n += 1
    assert n == 9
