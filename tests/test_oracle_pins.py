"""The oracle against closed forms, brute force and invariants (CPU only).

Both transcriptions of the forward definitions are pinned: the C loops
(``kdn_oracle.c``) by every pin, and the pure-Python loops
(``oracle.diag_scan_py`` / ``oracle.mobius_scan_py``) by the diagonal and
Moebius pins directly, plus a cross-check of the two on the smallest scan
workload (B=1, H=1, T=256, d=16, fp32 inputs)."""
import numpy as np
import pytest

import oracle
import oracle_pins
from bayesian_scan_gb300 import workloads


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("pin", oracle_pins.DIAG_PINS + oracle_pins.MOBIUS_PINS,
                         ids=lambda f: f.__name__)
def test_pin_pure_python(pin):
    pin(oracle_pins.PY)


def test_pure_python_equals_c_on_the_small_workload(oracle_lib):
    inp = workloads.make("small")
    args = [inp[n] for n in ("q", "k", "v", "beta", "d", "A")]
    rng = np.random.default_rng(5)
    w = workloads.get("small")
    I0 = 0.5 + rng.random((w.B, w.H, w.dv, w.dk))
    mu0 = rng.standard_normal((w.B, w.H, w.dv, w.dk))
    for state in ((None, None), (I0, mu0)):
        c = oracle.diag_scan(*args, inp["I_prior"], *state, lib=oracle_lib)
        p = oracle.diag_scan_py(*args, inp["I_prior"], *state)
        for x, r in zip(p, c):
            assert np.max(np.abs(x - r)) <= 1e-12 * np.max(np.abs(r))
    m = [inp[n] for n in ("ma", "mb", "mc", "md", "lam0")]
    c = oracle.mobius_scan(*m, lib=oracle_lib)
    p = oracle.mobius_scan_py(*m)
    assert np.max(np.abs(p - c)) <= 1e-12 * np.max(np.abs(c))
