"""Error model of the FP8 attention's P rounding -- TEST INFRASTRUCTURE.

The FP8 forward rounds the probabilities to OCP E4M3 before the P V product
while its row sum stays in fp32, so against attention of the dequantised
inputs (the oracle) each output element carries

    dO_id = sum_j e_j v_jd / l',   p'_j = 2^(x_j - m + 4),   l' = sum_j p'_j

with e_j the round-to-nearest error of p'_j on the E4M3 grid, whose spacing
at p'_j is q_j = 2^(max(floor(log2 p'_j), -6) - 3).  Modelling e_j as
independent and uniform on [-q_j/2, q_j/2] (variance q_j^2 / 12) gives

    sigma_id^2 = sum_j (q_j^2 / 12) v_jd^2 / l'^2.

The kernel's running maximum m lags the true row maximum by at most 4
(log2 units), which only moves p' up the grid (relatively finer); taking m
at the true maximum gives the largest sigma.  Tests accept
|dO| <= 7 sigma + bf16 output rounding + 1e-4.
"""
from __future__ import annotations

import numpy as np


def e4m3_spacing(p):
    """Spacing of the E4M3 grid at p >= 0 (2^-9 in the subnormal range; 0 at
    p = 0, which rounds without error)."""
    a = np.where(p > 0, p, 1.0)
    _, e = np.frexp(a)
    return np.where(p > 0, np.ldexp(1.0, np.maximum(e - 1, -6) - 3), 0.0)


def sigma_rows(q, k, v, rows, scale, block=256):
    """sigma[r, d] of the model above for query rows `rows` of one head.

    q, k, v: [N, D] arrays of the dequantised inputs (fp64 values)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v2 = np.asarray(v, dtype=np.float64) ** 2
    out = np.empty((len(rows), v2.shape[1]))
    log2e = 1.0 / np.log(2.0)
    for b0 in range(0, len(rows), block):
        r = rows[b0:b0 + block]
        x = (q[r] @ k.T) * (scale * log2e)
        x -= x.max(axis=1, keepdims=True)
        p = np.exp2(x + 4.0)
        l = p.sum(axis=1)
        w = e4m3_spacing(p) ** 2 / 12.0
        out[b0:b0 + block] = np.sqrt(w @ v2) / l[:, None]
    return out


def check_fp8(got_o, got_l, ref_o, ref_l, sigma, what=""):
    """Assert FP8 results agree with the oracle on the dequantised inputs."""
    go = np.asarray(got_o, dtype=np.float64)
    gl = np.asarray(got_l, dtype=np.float64)
    assert np.isfinite(go).all() and np.isfinite(gl).all(), f"{what}: non-finite output"
    bound = 7.0 * sigma + 2.0 ** -9 * np.abs(ref_o) + 1e-4
    err = np.abs(go - ref_o)
    worst = (err / bound).max() if err.size else 0.0
    assert worst <= 1.0, f"{what}: |dO| exceeds the E4M3 error model by {worst:.2f}x (max |dO| {err.max():.3e})"
    el = (np.abs(gl - ref_l) / np.maximum(np.abs(ref_l), 1e-30)).max() if gl.size else 0.0
    assert el <= 1e-3, f"{what}: max rel dLSE {el:.3e}"
    return float(err.max()) if err.size else 0.0, float(worst)
