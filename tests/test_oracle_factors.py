"""Pins of the fitted-factor reading of the compensators (LeapQuant §3.3 dominant
state components as rank-one terms; App. B.3, factors refitted at the boundary; research
note 4: eight power-iteration sweeps per compensator from the longest row),
against results the oracle does not compute itself."""
import numpy as np
import pytest

from oracle import FoldDiag, OracleState


def _rank2_plus_noise(seed, s1=40.0, s2=12.0, noise=1e-3):
    rng = np.random.default_rng(seed)
    u, _ = np.linalg.qr(rng.standard_normal((128, 2)))
    v, _ = np.linalg.qr(rng.standard_normal((128, 2)))
    S = s1 * np.outer(u[:, 0], v[:, 0]) + s2 * np.outer(u[:, 1], v[:, 1])
    S += noise * rng.standard_normal((128, 128))
    return S.astype(np.float32)


def test_factors_are_the_dominant_singular_components():
    """Power iteration from the longest row converges to the leading singular
    pairs; numpy's SVD is the independent reference."""
    S0 = _rank2_plus_noise(1)
    st = OracleState(1, C=2, comp_fit=8)
    dg = [FoldDiag(128, 128)]
    st.init(S0[None], diags=dg)
    U, sv, Vt = np.linalg.svd(S0.astype(np.float64))
    R1 = S0.astype(np.float64)
    for c in range(2):
        a = st.comp_line[0, c, :128].astype(np.float64)
        b = st.comp_line[0, c, 128:].astype(np.float64)
        assert abs(np.linalg.norm(b) - 1.0) < 1e-6
        sign = np.sign(b @ Vt[c])
        assert abs(abs(b @ Vt[c]) - 1.0) < 1e-6
        assert np.linalg.norm(a - sign * sv[c] * U[:, c]) <= 1e-4 * sv[c]
        R1 = R1 - np.outer(a, b)
    # what remains after both deflations is the noise
    assert np.linalg.norm(dg[0].R.astype(np.float64) - R1) <= 1e-5 * np.linalg.norm(S0)
    assert np.linalg.norm(dg[0].R) <= 3e-3 * 128


def test_deflated_residual_annihilates_the_fitted_direction():
    """(R - a b^T) b = R b - a (b . b) = 0 for the final a = R b and unit b."""
    rng = np.random.default_rng(2)
    S0 = (rng.standard_normal((128, 128)) * rng.uniform(0.1, 5, (128, 1))).astype(np.float32)
    st = OracleState(1, C=1, comp_fit=8)
    dg = [FoldDiag(128, 128)]
    st.init(S0[None], diags=dg)
    b = st.comp_line[0, 0, 128:].astype(np.float64)
    Rb = dg[0].R.astype(np.float64) @ b
    assert np.linalg.norm(Rb) <= 1e-5 * np.linalg.norm(S0.astype(np.float64) @ b)


def test_start_row_and_zero_state():
    S0 = np.zeros((2, 128, 128), np.float32)
    S0[1, 37, :] = 1.0
    S0[1, 90, :] = 0.5
    st = OracleState(2, C=2, comp_fit=8)
    st.init(S0)
    assert not st.comp_line[0].any()  # zero state: zero factors
    assert st.comp_id[1, 0] == 37     # the longest row starts the first fit
    np.testing.assert_allclose(st.comp_line[1, 0, 128:], np.full(128, 1 / np.sqrt(128)), rtol=1e-6)


@pytest.mark.parametrize("bits", [8, 4])
def test_half_step_reconstruction_with_factors(bits):
    """After every fold, dequantized residual plus the factor terms rebuild the
    state within half a step per entry (plus the deflation's own rounding)."""
    from quantized_linear_attention_gb300 import workload as wlm

    wl = wlm.WORKLOADS[2]
    N, W = 2, 16
    S0, _ = wlm.initial_state(wl, 0, N)
    tk = wlm.tokens(wl, 0, 2 * W, 0, N)
    st = OracleState(N, W=W, C=4, comp_fit=8, code_bits=bits)
    st.init(S0)
    for w in range(2):
        sl = slice(w * W, (w + 1) * W)
        st.run(tk.q[sl], tk.k[sl], tk.v[sl], tk.alpha[sl], tk.beta[sl], fold_when_full=False)
        dg = [FoldDiag(128, 128) for _ in range(N)]
        st.fold(diags=dg)
        for s in range(N):
            S = dg[s].S.astype(np.float64)
            step = st.sigma[s].astype(np.float64)[:, None] * st.lam[s].astype(np.float64)[None, :]
            rebuilt = st.dequant(s)
            slack = 8 * np.spacing(np.abs(S).max().astype(np.float32))
            assert np.all(np.abs(S - rebuilt) <= 0.5 * step * (1 + 1e-4) + slack)
