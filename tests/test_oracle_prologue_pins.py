"""Pins for the oracle's prologue functions (rotary embedding of q and k, the
projected V2 lambda), independent of their code:
  * rotary: position 0 is the identity; every row keeps its norm; a
    rotation by -p undoes one by p; q . k after rotation depends only on the
    distance of the two positions; the complex-number form (x_i + i x_{i+D/2})
    e^{i theta}; D = 2 rotates by exactly the position in radians;
  * lambda projection: one-hot tokens pick rows of w; numpy's matmul.
"""
import math

import numpy as np

from test_oracle_pins import rng_arrays


def test_rope_identity_norm_and_inverse(oracle):
    (x,) = rng_arrays(300, (2, 9, 3, 16))
    y = oracle.rope(x, pos0=0)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # a rotation by -p undoes one by p (row by row: T = 1 calls at each position)
    for t in range(x.shape[1]):
        fwd = oracle.rope(x[:, t:t + 1], pos0=37 + t)
        np.testing.assert_allclose(oracle.rope(fwd, pos0=-(37 + t)), x[:, t:t + 1], rtol=1e-12, atol=1e-13)


def test_rope_scores_depend_on_distance_only(oracle):
    q, k = rng_arrays(301, (1, 1, 1, 32), (1, 1, 1, 32))
    def score(m, n):
        return float((oracle.rope(q, pos0=m) * oracle.rope(k, pos0=n)).sum())
    for m, n, s in [(5, 2, 100), (0, 0, 7), (1000, 17, -17), (4, 9, 3000)]:
        assert abs(score(m, n) - score(m + s, n + s)) <= 1e-10 * max(1.0, abs(score(m, n)))
    assert abs(score(7, 3) - score(4, 3)) > 1e-6   # the distance does matter


def test_rope_complex_form_and_quarter_turn(oracle):
    B, T, H, D = 1, 6, 2, 8
    (x,) = rng_arrays(302, (B, T, H, D))
    base = 500.0
    y = oracle.rope(x, pos0=11, base=base)
    half = D // 2
    z = x[..., :half] + 1j * x[..., half:]
    pos = (11 + np.arange(T))[None, :, None, None]
    freq = base ** (-np.arange(half) / half)                    # base^(-2i/D)
    w = z * np.exp(1j * pos * freq)
    np.testing.assert_allclose(y[..., :half], w.real, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(y[..., half:], w.imag, rtol=1e-11, atol=1e-12)
    # D = 2: theta = the position itself (base^0 = 1), here 2 radians
    v = np.array([[[[0.3, -1.7]]]])
    r2 = oracle.rope(v, pos0=2)
    c, s = math.cos(2.0), math.sin(2.0)
    np.testing.assert_allclose(r2[0, 0, 0], [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], rtol=1e-14)


def test_lambda_proj_one_hot_and_library(oracle):
    C, P = 24, 5
    (w,) = rng_arrays(303, (C, P))
    x = np.zeros((2, 3, C))
    x[0, 0, 4] = 1.0
    x[1, 2, 23] = 1.0
    y = oracle.lambda_proj(x, w)
    np.testing.assert_array_equal(y[0, 0], w[4])
    np.testing.assert_array_equal(y[1, 2], w[23])
    np.testing.assert_array_equal(y[0, 1], np.zeros(P))
    (xr,) = rng_arrays(304, (4, 7, C))
    np.testing.assert_allclose(oracle.lambda_proj(xr, w), xr @ w, rtol=1e-12, atol=1e-12)
