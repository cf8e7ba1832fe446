"""Pins of the projection oracle (oracle/mixer.py) against facts that do not come from
it: brute-force sums on a tiny case, weights that select input coordinates (head split,
q/k/v order, the 1/sqrt(dk) scale), zero logits (beta = 1/2) and the logistic function
of the standard library."""
import math

import numpy as np

from oracle.mixer import mixer_proj


def test_brute_force_tiny():
    rng = np.random.default_rng(0)
    B, L, D, H, dk = 2, 3, 5, 2, 4
    x = rng.standard_normal((B, L, D))
    w = rng.standard_normal((3 * H * dk + H, D))
    q, k, v, beta = mixer_proj(x, w, H, dk)
    for b in range(B):
        for l in range(L):
            for h in range(H):
                for i in range(dk):
                    row = h * dk + i
                    s = [sum(x[b, l, d] * w[part * H * dk + row, d] for d in range(D)) for part in range(3)]
                    assert math.isclose(q[b, h, l, i], s[0] / math.sqrt(dk), rel_tol=1e-12, abs_tol=1e-12)
                    assert math.isclose(k[b, h, l, i], s[1], rel_tol=1e-12, abs_tol=1e-12)
                    assert math.isclose(v[b, h, l, i], s[2], rel_tol=1e-12, abs_tol=1e-12)
                z = sum(x[b, l, d] * w[3 * H * dk + h, d] for d in range(D))
                assert math.isclose(beta[b, h, l], 1.0 / (1.0 + math.exp(-z)), rel_tol=1e-12)


def test_selection_weights_fix_head_split_and_order():
    """W rows are unit vectors: q of head h, dim i reads x coordinate h*dk + i (scaled),
    k reads coordinate h*dk + i + 1 (mod D), v coordinate D - 1 - (h*dk + i)."""
    B, L, H, dk = 1, 4, 3, 8
    D = H * dk + 1
    x = np.arange(B * L * D, dtype=np.float64).reshape(B, L, D) / 7.0
    w = np.zeros((3 * H * dk + H, D))
    for r in range(H * dk):
        w[r, r] = 1.0
        w[H * dk + r, (r + 1) % D] = 1.0
        w[2 * H * dk + r, D - 1 - r] = 1.0
    q, k, v, beta = mixer_proj(x, w, H, dk)
    for h in range(H):
        for i in range(dk):
            r = h * dk + i
            np.testing.assert_array_equal(q[0, h, :, i], x[0, :, r] / math.sqrt(dk))
            np.testing.assert_array_equal(k[0, h, :, i], x[0, :, (r + 1) % D])
            np.testing.assert_array_equal(v[0, h, :, i], x[0, :, D - 1 - r])
    np.testing.assert_array_equal(beta, 0.5)          # zero logits


def test_beta_is_the_logistic_function():
    B, L, H, dk, D = 1, 6, 2, 4, 3
    x = np.linspace(-30, 30, B * L * D).reshape(B, L, D)
    w = np.zeros((3 * H * dk + H, D))
    w[3 * H * dk + 0, 0] = 1.0
    w[3 * H * dk + 1, 2] = -2.0
    _, _, _, beta = mixer_proj(x, w, H, dk)

    def logistic(z):   # tanh form for z >= 0, e^z / (1 + e^z) below (no cancellation either way)
        return 0.5 * (1 + math.tanh(z / 2)) if z >= 0 else math.exp(z) / (1 + math.exp(z))
    for l in range(L):
        z0, z1 = x[0, l, 0], -2.0 * x[0, l, 2]
        assert math.isclose(beta[0, 0, l], logistic(z0), rel_tol=1e-12)
        assert math.isclose(beta[0, 1, l], logistic(z1), rel_tol=1e-12)
