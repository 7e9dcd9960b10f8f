"""Pins for the rotary-embedding oracle (CPU only).

The tables are pinned by closed forms (angle = position at pair 0, the
geometric ratio theta^(-2/R) between neighbouring frequencies, angle
additivity in the position). The rotation is pinned against complex
multiplication z * exp(i angle), with the pairs read as complex numbers in the
two ways the pages use (numpy's own (re, im) layout for interleaved pairs, and
first half + i * second half for the half-split pairing), by norm preservation,
the relative-position property of the inner product, and the permutation that
maps one pairing onto the other. A mutation test plants mistakes in copies of
the oracle and checks that a pin catches each.
"""
import numpy as np
import pytest

from oracle import rope

THETA = 10000.0


def _rand(shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


def test_tables_closed_forms():
    for R in (8, 64, 128):
        cos, sin = rope.tables(THETA, 40, R)
        p = np.arange(40)
        np.testing.assert_allclose(cos[:, 0], np.cos(p), atol=1e-15)
        np.testing.assert_allclose(sin[:, 0], np.sin(p), atol=1e-15)
        np.testing.assert_array_equal(cos[0], 1.0)
        np.testing.assert_array_equal(sin[0], 0.0)
        # neighbouring frequencies: the angle at position 1 shrinks by theta^(-2/R) per pair
        ang1 = np.arctan2(sin[1], cos[1])
        np.testing.assert_allclose(ang1[1:] / ang1[:-1], THETA ** (-2.0 / R), rtol=1e-12)


def test_tables_angle_additivity():
    cos, sin = rope.tables(THETA, 64, 64)
    for a, b in ((3, 5), (17, 30), (1, 62)):
        np.testing.assert_allclose(cos[a + b], cos[a] * cos[b] - sin[a] * sin[b], atol=1e-12)
        np.testing.assert_allclose(sin[a + b], sin[a] * cos[b] + cos[a] * sin[b], atol=1e-12)


def _complex_reference(x, pos, cos, sin, R, interleaved):
    tokens, rows, width = x.shape
    seg = x.reshape(tokens, rows, width // R, R)
    if interleaved:
        z = np.ascontiguousarray(seg).view(np.complex128)          # (re, im) = (2i, 2i+1)
    else:
        z = seg[..., : R // 2] + 1j * seg[..., R // 2:]
    rot = (cos[pos] + 1j * sin[pos])[:, None, None, :]
    w = z * rot
    if interleaved:
        out = np.ascontiguousarray(w).view(np.float64)
    else:
        out = np.concatenate([w.real, w.imag], axis=-1)
    return out.reshape(tokens, rows, width)


@pytest.mark.parametrize("R,interleaved", [(16, True), (16, False), (32, False), (32, True)])
def test_rotation_is_complex_multiplication(R, interleaved):
    x = _rand((11, 3, 32), 1)
    pos = np.random.default_rng(2).integers(0, 50, 11)
    cos, sin = rope.tables(THETA, 50, R)
    got = rope.apply(x, pos, cos, sin, R, interleaved)
    np.testing.assert_allclose(got, _complex_reference(x, pos, cos, sin, R, interleaved), atol=1e-13)


def test_norm_preserved_and_position_zero_identity():
    x = _rand((5, 2, 64), 3)
    cos, sin = rope.tables(THETA, 20, 64)
    for inter in (True, False):
        y = rope.apply(x, np.array([0, 3, 7, 11, 19]), cos, sin, 64, inter)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(y[0], x[0], atol=0)


def test_relative_position_property():
    """<R(p) q, R(p') k> depends on p - p' only."""
    q, k = _rand((1, 1, 64), 4), _rand((1, 1, 64), 5)
    cos, sin = rope.tables(THETA, 200, 64)
    for inter in (True, False):
        def dot(p, pk):
            return float((rope.apply(q, [p], cos, sin, 64, inter) * rope.apply(k, [pk], cos, sin, 64, inter)).sum())
        base = dot(10, 3)
        for s in (1, 40, 150):
            assert abs(dot(10 + s, 3 + s) - base) < 1e-10
        assert abs(dot(11, 3) - base) > 1e-6


def test_pairings_related_by_permutation():
    R = 16
    perm = np.concatenate([np.arange(0, R, 2), np.arange(1, R, 2)])  # interleaved -> half layout
    x = _rand((6, 2, R), 6)
    pos = np.arange(6) * 3
    cos, sin = rope.tables(THETA, 20, R)
    inter = rope.apply(x, pos, cos, sin, R, True)
    half = rope.apply(x[..., perm], pos, cos, sin, R, False)
    np.testing.assert_allclose(half, inter[..., perm], atol=1e-14)


def test_segments_are_independent():
    """Rotary width d on a 2d-wide head row = each d-wide component on its own."""
    x = _rand((4, 3, 32), 7)
    cos, sin = rope.tables(THETA, 10, 16)
    pos = [1, 4, 2, 9]
    whole = rope.apply(x, pos, cos, sin, 16, False)
    for c in range(2):
        part = rope.apply(x[..., c * 16:(c + 1) * 16], pos, cos, sin, 16, False)
        np.testing.assert_allclose(whole[..., c * 16:(c + 1) * 16], part, atol=0)


def test_half_pairing_crosses_components_at_full_width():
    """At R = 2d with the half pairing, coordinate i of q1 pairs with coordinate i of
    q2 (the Llama placement): rotating [q1 | 0] moves energy into the q2 half."""
    x = np.zeros((1, 1, 32))
    x[0, 0, :16] = _rand((16,), 8)
    cos, sin = rope.tables(THETA, 4, 32)
    y = rope.apply(x, [3], cos, sin, 32, False)
    assert np.abs(y[0, 0, 16:]).sum() > 0.1


def test_positions_from_cu_seqlens():
    np.testing.assert_array_equal(rope.positions_from_cu_seqlens([0, 3, 3, 5]), [0, 1, 2, 0, 1])


def _mutants():
    def sign(x, positions, cos, sin, R, inter):
        return rope.apply(x, positions, cos, -sin, R, inter)

    def swapped(x, positions, cos, sin, R, inter):
        return rope.apply(x, positions, cos, sin, R, not inter)

    def off_by_one(x, positions, cos, sin, R, inter):
        return rope.apply(x, np.asarray(positions) + 1, cos, sin, R, inter)

    def transposed(x, positions, cos, sin, R, inter):
        return rope.apply(x, positions, sin, cos, R, inter)
    return [sign, swapped, off_by_one, transposed]


@pytest.mark.parametrize("mutant", _mutants())
def test_mutants_are_caught(mutant):
    x = _rand((7, 2, 32), 9)
    pos = np.array([0, 1, 2, 5, 8, 13, 21])
    cos, sin = rope.tables(THETA, 30, 32)
    for inter in (True, False):
        ref = _complex_reference(x, pos, cos, sin, 32, inter)
        if not np.allclose(mutant(x, pos, cos, sin, 32, inter), ref, atol=1e-9):
            return
    pytest.fail("mutant not caught")


def test_wrong_frequency_exponent_is_caught():
    cos, sin = rope.tables(THETA, 5, 64)
    i = np.arange(32)
    bad = np.cos(np.arange(5)[:, None] * THETA ** (-i / 64.0))
    ang1 = np.arctan2(np.sin(np.arange(5)[:, None] * THETA ** (-i / 64.0)), bad)[1]
    assert not np.allclose(ang1[1:] / ang1[:-1], THETA ** (-2.0 / 64))
