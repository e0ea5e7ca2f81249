"""Pins for the oracle's rotary re-alignment: closed forms and group laws of
plane rotations, independent of the oracle's own code path."""
import math

import numpy as np
import pytest

import oracle


def test_hand_computed_pairs_interleaved():
    # d = 4, rotary_dim = 4, base 100: theta = (1, 1/10)
    x = np.array([[1.0, 0.0, 0.0, 1.0]])
    d = 0.7
    y = oracle.rope(x, [d], 4, 0, 100.0)
    want = [math.cos(d), math.sin(d), -math.sin(d / 10), math.cos(d / 10)]
    np.testing.assert_allclose(y[0], want, rtol=0, atol=1e-15)


def test_hand_computed_pairs_split_half():
    # style 1 pairs (0, 2) and (1, 3)
    x = np.array([[2.0, 0.0, 0.0, 3.0]])
    d = 1.3
    y = oracle.rope(x, [d], 4, 1, 100.0)
    want = [2 * math.cos(d), -3 * math.sin(d / 10), 2 * math.sin(d), 3 * math.cos(d / 10)]
    np.testing.assert_allclose(y[0], want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("style", [0, 1])
def test_composition_inverse_identity_and_norms(style):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 128))
    p, dlt = rng.integers(0, 100000, 50).astype(float), 3789.0
    a = oracle.rope(oracle.rope(x, p, 96, style, 10000.0), [dlt] * 50, 96, style, 10000.0)
    b = oracle.rope(x, p + dlt, 96, style, 10000.0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)
    back = oracle.rope(oracle.rope(x, p, 96, style, 10000.0), -p, 96, style, 10000.0)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-9)
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(50), 96, style, 10000.0), x)
    y = oracle.rope(x, p, 96, style, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_array_equal(y[:, 96:], x[:, 96:])  # beyond rotary_dim untouched


def test_relative_position_invariance_of_scores():
    # q.k after rotating both to (p+t, p) depends only on t (the RoPE property)
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    s = [float((oracle.rope(q, [p + 5], 64, 0, 10000.0) @ oracle.rope(k, [p], 64, 0, 10000.0).T)[0, 0])
         for p in (0, 17, 4096)]
    np.testing.assert_allclose(s, s[0], rtol=0, atol=1e-10)
