"""The FP8 error model against a simulation of the kernel's arithmetic on the
CPU: P rounded to E4M3 by the oracle's rounding (independent of the error
model's grid-spacing formula), row sums of the unrounded P.  The model's
7-sigma bound must hold for every element and its sigma must predict the
observed RMS error within a factor of two."""
import numpy as np

import oracle
from tests.fp8_error_model import e4m3_spacing, sigma_rows


def test_spacing_matches_the_e4m3_grid():
    """At every positive E4M3 value the model's spacing is the gap to the next
    value, with the grid decoded from the format's bit fields."""
    vals = []
    for code in range(127):                                  # positive codes, NaN (127) excluded
        e, m = code >> 3, code & 7
        vals.append((m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    vals = np.array(sorted(vals))
    np.testing.assert_array_equal(e4m3_spacing(vals[1:-1]), np.diff(vals)[1:])
    assert e4m3_spacing(np.array([0.0]))[0] == 0.0


def test_model_bounds_simulated_fp8_rounding():
    rng = np.random.default_rng(41)
    N, D, scale = 3000, 64, 1 / 8
    q, k, v = (rng.standard_normal((n, D)) for n in (200, N, N))
    rows = np.arange(200)
    x = (q @ k.T) * (scale / np.log(2.0))
    for lag in (0.0, 2.5):                                   # running maximum at or below the true one
        m = x.max(axis=1, keepdims=True) - lag
        pp = np.exp2(x - m + 4.0)
        l = pp.sum(axis=1, keepdims=True)
        exact = (pp @ v) / l
        fp8 = (oracle.e4m3_round(pp) @ v) / l
        err = np.abs(fp8 - exact)
        sig = sigma_rows(q, k, v, rows, scale)
        assert np.all(err <= 7 * sig + 1e-12)
        ratio = np.sqrt((err ** 2).mean()) / np.sqrt((sig ** 2).mean())
        assert ratio < 2.0
        if lag == 0.0:
            assert ratio > 0.5                               # the model is not vacuous
