"""Pins for the output-projection oracle (CPU only): brute-force sums on small
non-square shapes (which also catch a transposed weight), the [tokens, H, dv]
input flattening in head-major order, and identity / zero weights."""
import numpy as np

from oracle import out_proj as oo


def test_brute_force_non_square():
    rng = np.random.default_rng(0)
    x, w = rng.standard_normal((5, 7)), rng.standard_normal((3, 7))
    want = np.zeros((5, 3))
    for t in range(5):
        for n in range(3):
            for k in range(7):
                want[t, n] += x[t, k] * w[n, k]
    np.testing.assert_allclose(oo.out_proj(x, w), want, atol=1e-12)


def test_head_major_flattening():
    """Column h * dv + j of the flattened input is head h, value j."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 3, 2))
    w = np.zeros((1, 6))
    w[0, 1 * 2 + 1] = 1.0
    np.testing.assert_array_equal(oo.out_proj(x, w)[:, 0], x[:, 1, 1])


def test_identity_and_zero():
    x = np.random.default_rng(2).standard_normal((6, 4))
    np.testing.assert_array_equal(oo.out_proj(x, np.eye(4)), x)
    np.testing.assert_array_equal(oo.out_proj(x, np.zeros((2, 4))), np.zeros((6, 2)))
