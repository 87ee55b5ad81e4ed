"""Pins of the block fit of the compensator factors (reading R25).

The research note's redesign fits the C compensators together as a block,
starting from the previous window's compensators, and gives a counterexample
where a start from the longest row misses the strongest pattern that a block
fit captures (fastpathlabs.ai research note 4, "Where the time goes" and
"Redesign"). The oracle's block fit is subspace iteration; it is pinned here
against numpy's SVD and against the algebra of deflation, not against itself.
"""
import numpy as np
import pytest

from oracle import fit


def _matrix(rng, sig, dv=128, dk=128):
    U, _ = np.linalg.qr(rng.standard_normal((dv, dv)))
    V, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    s = np.zeros(min(dv, dk))
    s[:len(sig)] = sig
    return (U[:, :len(s)] * s) @ V.T[:len(s)], U, V


def _proj(B):
    return B.T @ B


def test_block_fit_finds_the_leading_right_singular_subspace():
    rng = np.random.default_rng(11)
    sig = np.concatenate([[40, 30, 20, 10], np.linspace(1.0, 0.1, 124)])
    R, U, V = _matrix(rng, sig)
    a, b, ids, Rd = fit(R, 4, 40, block=True)
    assert ids.tolist() == [0, 1, 2, 3]
    assert np.abs(b @ b.T - np.eye(4)).max() < 1e-5  # orthonormal
    assert np.abs(_proj(b) - V[:, :4] @ V[:, :4].T).max() < 1e-4  # the top-4 subspace
    # a_c = R_c b_c on the residual left by the earlier factors; with b orthonormal
    # that is R b_c, and the deflated residual has no component along span(b)
    R64 = R.astype(np.float64)
    assert np.abs(a - (R64 @ b.T).T).max() < 1e-3 * np.abs(a).max()
    assert np.linalg.norm(Rd.astype(np.float64) @ b.T) < 1e-4 * np.linalg.norm(R64)
    # captured energy = the top-4 singular values squared
    assert abs((a.astype(np.float64) ** 2).sum() - (sig[:4] ** 2).sum()) < 1e-3 * (sig[:4] ** 2).sum()


def test_warm_start_from_the_exact_factors_is_a_fixed_point():
    rng = np.random.default_rng(12)
    sig = np.concatenate([[9, 7, 5], np.linspace(0.5, 0.05, 125)])
    R, U, V = _matrix(rng, sig)
    prev_b = V[:, :3].T.astype(np.float32)
    prev_a = (U[:, :3] * sig[:3]).T.astype(np.float32)
    a, b, _, _ = fit(R, 3, 1, block=True, prev=(prev_a, prev_b))
    for c in range(3):
        assert abs(abs(float(b[c] @ V[:, c])) - 1.0) < 1e-5
        assert np.linalg.norm(np.abs(a[c]) - sig[c] * np.abs(U[:, c])) < 1e-4 * sig[c]


def _counterexample(rng):
    """The longest row points along e0 (length 10); a hundred shorter rows point along
    e1 (length 2 each), so the strongest pattern is e1 (energy 400 against 100). The
    two patterns are exactly orthogonal, so a fit that starts on e0 stays there."""
    R = np.zeros((128, 128), np.float32)
    R[0, 0] = 10.0
    R[1:101, 1] = 2.0
    R[101:, 2:] = (1e-3 * rng.standard_normal((27, 126))).astype(np.float32)  # weak, elsewhere
    return R


def test_the_longest_row_start_misses_what_the_block_fit_captures():
    rng = np.random.default_rng(13)
    R = _counterexample(rng)
    a1, b1, _, _ = fit(R, 1, 8, block=False)  # one at a time, from the longest row
    assert abs(b1[0, 0]) > 0.999 and (a1.astype(np.float64) ** 2).sum() == pytest.approx(100.0, rel=1e-3)
    start_b = np.zeros((1, 128), np.float32)
    start_b[0, :2] = np.float32(np.sqrt(0.5))  # a previous factor that overlaps both patterns
    a2, b2, _, _ = fit(R, 1, 8, block=True, prev=(np.zeros((1, 128), np.float32), start_b))
    assert abs(b2[0, 1]) > 0.999 and (a2.astype(np.float64) ** 2).sum() == pytest.approx(400.0, rel=1e-3)


def test_zero_previous_factors_fall_back_to_the_longest_rows():
    rng = np.random.default_rng(14)
    R = _counterexample(rng)
    zero = (np.zeros((2, 128), np.float32), np.zeros((2, 128), np.float32))
    a, b, _, _ = fit(R, 2, 1, block=True, prev=zero)
    a_cold, b_cold, _, _ = fit(R, 2, 1, block=True)
    assert np.array_equal(b, b_cold) and np.array_equal(a, a_cold)
    # started from row 0 (e0), then the first e1 row: one sweep keeps that order
    assert abs(b[0, 0]) > 0.999 and abs(b[1, 1]) > 0.999


def test_rank_deficient_block_keeps_a_zero_factor():
    """Where the start vectors are dependent, Gram-Schmidt leaves a zero factor, and a
    zero factor stays zero (its term is exactly 0)."""
    R = np.zeros((128, 128), np.float32)
    R[:, 3] = 1.0  # rank one: every row is e3
    a, b, _, Rd = fit(R, 2, 4, block=True)
    assert abs(b[0, 3]) == pytest.approx(1.0, abs=1e-6)
    assert not b[1].any() and not a[1].any()
    assert np.abs(Rd).max() < 1e-5
