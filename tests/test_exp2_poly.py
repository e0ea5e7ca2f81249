"""The softmax's base-2 exponential on the FMA pipe (exp2_poly in csrc/ptx.cuh).

2^x = 2^i * 2^f with i the nearest integer and f in [-1/2, 1/2]; 2^f is a
cubic whose coefficients the library states as constants. They are pinned
here to mathematics, independently of the library:
  - on the CPU, a Remez exchange on the relative error written in this file
    re-derives the minimax cubic for 2^f on [-1/2, 1/2], and the library's
    constants must equal it; its error must equioscillate at five points with
    magnitude 7.48e-5 (Chebyshev's alternation theorem);
  - on the GPU, the device function itself (through segkv_exp2_check) must be
    within that bound plus fp32 rounding of fp64 2^x on a dense grid of
    [-125, 0] (the softmax passes at most 8; [0, 8] is the same cubic shifted
    by whole exponents), and must give 2^-125 below -125, -inf included,
    within the cubic's bound, as stated.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUND = 7.48e-5


def library_coefficients():
    src = open(os.path.join(ROOT, "head_segmented_paged_gb300", "csrc", "ptx.cuh")).read()
    body = src[src.index("float exp2_poly(float x)"):]
    got = dict(re.findall(r"(c[0-3]) = ([0-9.]+)f", body[:600]))
    return np.array([float(got[f"c{k}"]) for k in range(4)])  # c0 .. c3


def remez_cubic_exp2(iters=20):
    """Minimax cubic for 2^f on [-1/2, 1/2] in the relative error: solve
    p(x_i) / 2^x_i - 1 = (-1)^i E on five reference points, move them to the
    error's extrema, repeat."""
    grid = np.linspace(-0.5, 0.5, 400001)
    x = 0.5 * np.cos(np.pi * np.arange(5)[::-1] / 4)
    for _ in range(iters):
        A = np.zeros((5, 5))
        A[:, :4] = x[:, None] ** np.arange(4)
        A[:, 4] = -((-1.0) ** np.arange(5)) * np.exp2(x)
        sol = np.linalg.solve(A, np.exp2(x))
        c, E = sol[:4], sol[4]
        err = np.polynomial.polynomial.polyval(grid, c) / np.exp2(grid) - 1
        turn = np.where(np.diff(np.sign(np.diff(err))) != 0)[0] + 1
        pts = np.concatenate([[0], turn, [grid.size - 1]])
        assert pts.size == 5
        x = grid[pts]
    return c, abs(E)


def test_library_cubic_is_the_minimax_cubic():
    c_lib = library_coefficients()
    c_ref, E = remez_cubic_exp2()
    np.testing.assert_allclose(c_lib, c_ref, rtol=2e-7, atol=0)
    assert abs(E - 7.478e-5) < 1e-8


def test_library_cubic_equioscillates_within_its_bound():
    c = library_coefficients()
    f = np.linspace(-0.5, 0.5, 1000001)
    err = np.polynomial.polynomial.polyval(f, c) / np.exp2(f) - 1
    assert np.abs(err).max() <= BOUND
    turn = np.where(np.diff(np.sign(np.diff(err))) != 0)[0] + 1
    ext = np.concatenate([[err[0]], err[turn], [err[-1]]])
    assert ext.size == 5
    assert (np.sign(ext[1:]) == -np.sign(ext[:-1])).all()  # alternating signs
    assert np.abs(ext).min() > 0.999 * np.abs(ext).max()   # equal magnitudes


def test_a_wrong_coefficient_is_caught():
    c = library_coefficients().copy()
    c[2] *= 1.001  # one coefficient off by 0.1 %
    f = np.linspace(-0.5, 0.5, 100001)
    err = np.polynomial.polynomial.polyval(f, c) / np.exp2(f) - 1
    assert np.abs(err).max() > BOUND


@pytest.mark.gpu
def test_device_exp2_poly_against_fp64():
    import torch

    import head_segmented_paged_gb300 as S

    rng = np.random.default_rng(0)
    xs = np.concatenate([
        np.linspace(-125.0, 8.0, 2_000_001),
        rng.uniform(-125.0, 0.0, 1_000_000),
        -(np.arange(0, 125) + 0.5),  # half-integers: f = +-1/2, the interval ends
        -np.arange(0, 126, dtype=np.float64),  # integers: f = 0, exact powers
    ]).astype(np.float32)
    below = np.array([-125.5, -126.0, -200.0, -1e30, -np.inf], np.float32)
    x = torch.from_numpy(np.concatenate([xs, below])).cuda()
    yp = torch.empty_like(x)
    ym = torch.empty_like(x)
    assert S.segkv_exp2_check(x, yp, ym) == 0
    torch.cuda.synchronize()
    yp, ym = yp.cpu().numpy().astype(np.float64), ym.cpu().numpy().astype(np.float64)
    n = xs.size
    exact = np.exp2(xs.astype(np.float64))
    rel = np.abs(yp[:n] / exact - 1)
    # the cubic's bound plus fp32 rounding of three FMAs and the result
    assert rel.max() <= BOUND + 4 * 2.0 ** -24, rel.max()
    # and against the hardware ex2 (its own error is a few fp32 ulps)
    rel_hw = np.abs(yp[:n] / ym[:n] - 1)
    assert rel_hw.max() <= BOUND + 2.0 ** -20, rel_hw.max()
    # below -125, -inf included: clamped to -125, so 2^-125 within the cubic's
    # bound (its value at f = 0 is c0, not exactly 1); the hardware gives 0 at -inf
    nb = below.size
    assert (np.abs(yp[n:n + nb] / 2.0 ** -125 - 1) <= BOUND + 4 * 2.0 ** -24).all()
    assert ym[n + nb - 1] == 0.0
