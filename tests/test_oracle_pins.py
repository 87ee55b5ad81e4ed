"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test checks the oracle against something other than itself: the plain
per-token recurrence in float64 (PIN-1), a separately written naive per-token
quantizer (PIN-2), hand-expanded products on d = 4 (PIN-3), the half-step
reconstruction bound (PIN-4), planted outlier lines (PIN-5), the associative
memory closed form (PIN-6), idempotence at beta = 0 (PIN-7), power-of-two scale
invariance (PIN-9), the textbook per-row absmax quantizer, the smoothing formula
and exact dot products.
"""
from __future__ import annotations

import fractions
import math

import numpy as np
import pytest

import oracle
from oracle import FoldDiag, OracleState
from quantized_linear_attention_gb300 import workload as wlm
from tests._helpers import code_mismatches, near_tie, rel_l2, selection_ties, tie_rows


# ---------------------------------------------------------------- dot products
@pytest.mark.parametrize("d", [4, 16, 128, 32])
def test_dot_within_fp32_error_bound_of_exact(d):
    rng = np.random.default_rng(d)
    for _ in range(50):
        a = rng.standard_normal(d).astype(np.float32)
        b = rng.standard_normal(d).astype(np.float32)
        exact = sum(fractions.Fraction(float(x)) * fractions.Fraction(float(y)) for x, y in zip(a, b))
        got = oracle.dot(a, b)
        bound = (d + 8) * 2.0**-24 * float(np.sum(np.abs(a.astype(np.float64) * b)))
        assert abs(got - float(exact)) <= bound


def test_sum_abs_within_bound():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(128).astype(np.float32)
    exact = math.fsum(abs(float(x)) for x in a)
    assert abs(oracle.sum_abs(a) - exact) <= 140 * 2.0**-24 * exact


def test_dot_is_exact_on_integers():
    a = np.arange(-64, 64, dtype=np.float32)
    b = np.arange(128, dtype=np.float32)[::-1].copy()
    assert oracle.dot(a, b) == float(np.dot(a.astype(np.int64), b.astype(np.int64)))


# ---------------------------------------------------------------- PIN-1
def _plain_recurrence(S0, tk, kda):
    """Plain per-token delta rule in float64 (LeapQuant §3.1 / App. A):
    u_t = beta_t (v_t - S_{t-1}(alpha_t . k_t)); S_t = S_{t-1} Diag(alpha_t) + u_t k_t^T; o_t = S_t q_t."""
    S = S0.astype(np.float64).copy()
    T = tk.q.shape[0]
    outs, states = [], []
    for t in range(T):
        q, k, v = (x[t].astype(np.float64) for x in (tk.q, tk.k, tk.v))
        a = tk.alpha[t].astype(np.float64)
        a = a if kda else a[:, None] * np.ones_like(k)
        beta = tk.beta[t].astype(np.float64)
        r = np.einsum("nij,nj->ni", S, a * k)
        u = beta[:, None] * (v - r)
        S = S * a[:, None, :] + u[:, :, None] * k[:, None, :]
        outs.append(np.einsum("nij,nj->ni", S, q))
        states.append(S.copy())
    return np.stack(outs), states


@pytest.mark.parametrize("case", ["gdn_zero_start", "gdn_warm_planted", "kda_t3"])
def test_pin1_windowed_unquantized_equals_plain_recurrence(case):
    if case == "gdn_zero_start":
        wl = wlm.WORKLOADS[1]
        N, T = 2, 64
        S0 = np.zeros((N, 128, 128), np.float32)
        tk = wlm.tokens(wl, 0, T)
    elif case == "gdn_warm_planted":
        wl = wlm.WORKLOADS[2]
        N, T = 3, 40
        S0, _ = wlm.initial_state(wl, 0, N)
        tk = wlm.tokens(wl, 0, T, 0, N)
    else:
        wl = wlm.WORKLOADS[5]
        N, T = 2, 40
        S0, _ = wlm.initial_state(wl, 0, N)
        tk = wlm.tokens(wl, 0, T, 0, N)
    W = 16
    st = OracleState(N, W=W, C=0, decay_per_key=wl.kda, quantize=False)
    st.init(S0)
    o_ref, S_ref = _plain_recurrence(S0, tk, wl.kda)
    o = np.zeros_like(o_ref)
    for t in range(T):
        o[t] = st.run(*(x[t:t + 1] for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta)))[0]
        S_now = st.export()  # boundary + records (or the new boundary right after a fold)
        err = rel_l2(S_now.reshape(N, -1), S_ref[t].reshape(N, -1))
        assert err.max() <= 1e-5, (t, err)
        if (t + 1) % W == 0:
            assert (st.count == 0).all()
            assert rel_l2(st.B.reshape(N, -1), S_ref[t].reshape(N, -1)).max() <= 1e-5
    assert rel_l2(o, o_ref).max() <= 1e-5


# ---------------------------------------------------------------- PIN-2
@pytest.mark.parametrize("bits", [8, 6, 4])
def test_pin2_window1_no_comp_no_smooth_is_naive_per_token_rounding(bits):
    """W = 1, C = 0, smoothing off is the naive scheme: round after every token
    (research note 4, "Why rounding the state is difficult"), at 8-, 6- and
    4-bit codes (LeapQuant §4). The naive side is written here in numpy float32,
    independently; compared in lockstep."""
    qm = 2 ** (bits - 1) - 1
    wl = wlm.custom(101, 4, 48, n_warm=64)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, wl.n_tokens)
    st = OracleState(wl.n_states, W=1, C=0, smooth=False, code_bits=bits)
    st.init(S0)
    f32 = np.float32
    total = 0
    for t in range(wl.n_tokens):
        q, k, v, a, beta = tk.token(t)
        codes0, sig0 = st.codes.copy(), st.sigma.copy()
        Sprev = sig0[:, :, None] * codes0.astype(f32)  # dequantize
        ak = (a[:, None] * k).astype(f32)
        r = np.einsum("nij,nj->ni", Sprev.astype(np.float64), ak.astype(np.float64)).astype(f32)
        u = (beta[:, None] * (v - r)).astype(f32)
        Snew = (a[:, None, None] * Sprev + u[:, :, None] * k[:, None, :]).astype(f32)
        m = np.abs(Snew).max(axis=2)
        h = np.where(m > 0, f32(qm) / np.where(m > 0, m, 1), 0).astype(f32)
        s = (Snew * h[:, :, None]).astype(f32)
        codes_naive = np.clip(np.rint(s), -qm, qm).astype(np.int8)
        o_naive = np.einsum("nij,nj->ni", Snew.astype(np.float64), q.astype(np.float64))

        o = st.run(q[None], k[None], v[None], a[None], beta[None])[0]
        assert rel_l2(o, o_naive).max() <= 1e-5
        n, ok = code_mismatches(st.codes, codes_naive, s, rel=0.0, abs_=1e-4)
        assert ok, t
        total += n
        np.testing.assert_allclose(st.sigma, m / f32(qm), rtol=3e-7, atol=0)
        assert np.abs(st.codes).max() <= qm
    assert total <= 1e-3 * wl.n_tokens * st.codes.size


# ---------------------------------------------------------------- PIN-3
def _dequant64(st, s=0):
    return st.dequant(s)


@pytest.mark.parametrize("kda", [False, True])
def test_pin3_d4_brute_force(kda):
    """d = 4, W = 3, C = 1, smoothing on: selection by enumerating all 8 lines,
    smoothing and scales by their formulas, three tokens by hand-expanded products."""
    S0 = np.array([[0.30, -0.20, 4.00, 0.10],
                   [-0.10, 0.25, -3.50, 0.05],
                   [0.20, 0.15, 5.00, -0.30],
                   [0.05, -0.40, -4.50, 0.20]], np.float32)
    floor = 1e-6
    st = OracleState(1, dk=4, dv=4, W=3, C=1, decay_per_key=kda, smooth=True, lambda_floor=floor)
    dg = [FoldDiag(4, 4)]
    st.init(S0[None], diags=dg)
    S64 = S0.astype(np.float64)
    scores = [float((S64[i] ** 2).sum()) for i in range(4)] + [float((S64[:, j] ** 2).sum()) for j in range(4)]
    best = int(np.argmax(scores))
    assert best == 4 + 2  # column 2 holds the outliers
    assert st.comp_id[0, 0] == best
    assert np.array_equal(st.comp_line[0, 0, :4], S0[:, 2])
    R = S64.copy()
    R[:, 2] = 0.0
    lam = np.maximum(np.sqrt(np.abs(R).mean(axis=0)), floor)
    np.testing.assert_allclose(st.lam[0], lam, rtol=2e-7)
    t = R / lam[None, :]
    sig = np.abs(t).max(axis=1) / 127.0
    np.testing.assert_allclose(st.sigma[0], sig, rtol=5e-7)
    s_ref = t / sig[:, None]
    assert not near_tie(s_ref, rel=1e-5).any()
    assert np.array_equal(st.codes[0], np.rint(s_ref).astype(np.int8))

    B = _dequant64(st)
    q = np.array([[0.5, -0.5, 0.5, 0.5], [0.1, 0.7, -0.7, 0.1], [-0.6, 0.0, 0.8, 0.0]], np.float32)
    k = np.array([[0.0, 0.6, 0.8, 0.0], [0.5, 0.5, 0.5, 0.5], [0.8, 0.0, 0.0, -0.6]], np.float32)
    v = np.array([[1.0, -2.0, 0.5, 3.0], [-1.0, 0.25, 2.0, -0.5], [0.75, 1.5, -1.25, 0.0]], np.float32)
    if kda:
        al = np.array([[0.9, 0.5, 0.8, 0.7], [0.6, 0.95, 0.85, 0.75], [0.99, 0.65, 0.55, 0.9]], np.float32)
    else:
        al = np.array([0.9, 0.8, 0.85], np.float32)
    beta = np.array([0.6, 0.3, 0.9], np.float32)
    f = lambda x: x.astype(np.float64)  # noqa: E731
    a1, a2, a3 = (f(al[i]) * np.ones(4) for i in range(3))
    k1, k2, k3 = f(k[0]), f(k[1]), f(k[2])
    v1, v2, v3 = f(v[0]), f(v[1]), f(v[2])
    b1, b2, b3 = (float(x) for x in beta)
    D = np.diag
    u1 = b1 * (v1 - B @ (a1 * k1))
    S1 = B @ D(a1) + np.outer(u1, k1)
    u2 = b2 * (v2 - (B @ D(a1) + np.outer(u1, k1)) @ (a2 * k2))
    S2 = (B @ D(a1) + np.outer(u1, k1)) @ D(a2) + np.outer(u2, k2)
    u3 = b3 * (v3 - ((B @ D(a1) + np.outer(u1, k1)) @ D(a2) + np.outer(u2, k2)) @ (a3 * k3))
    S3 = ((B @ D(a1) + np.outer(u1, k1)) @ D(a2) + np.outer(u2, k2)) @ D(a3) + np.outer(u3, k3)
    o_ref = [S1 @ f(q[0]), S2 @ f(q[1]), S3 @ f(q[2])]
    alpha_in = al[:, None, :] if kda else al[:, None]
    for t in range(3):
        o = st.run(q[t][None, None], k[t][None, None], v[t][None, None], alpha_in[t][None], beta[t:t + 1][None],
                   fold_when_full=False)[0, 0]
        assert rel_l2(o, o_ref[t]) <= 1e-6
    np.testing.assert_allclose(st.rec_u[0], np.stack([u1, u2, u3]), rtol=1e-5, atol=1e-6)
    dg2 = [FoldDiag(4, 4)]
    st.fold(diags=dg2)
    assert rel_l2(dg2[0].S.ravel(), S3.ravel()) <= 1e-6
    assert st.count[0] == 0


# ---------------------------------------------------------------- PIN-4
@pytest.mark.parametrize("wid", [1, 5])
@pytest.mark.parametrize("bits", [8, 4])
def test_pin4_half_step_reconstruction_after_every_fold(wid, bits):
    wl = wlm.WORKLOADS[wid]
    N = 2
    W = wl.W
    S0, _ = wlm.initial_state(wl, 0, N)
    tk = wlm.tokens(wl, 0, 3 * W, 0, N)
    st = OracleState(N, W=W, C=4, decay_per_key=wl.kda, code_bits=bits)
    dg0 = [FoldDiag(128, 128) for _ in range(N)]
    st.init(S0, diags=dg0)
    folds = [dg0]
    for w in range(3):
        sl = slice(w * W, (w + 1) * W)
        st.run(tk.q[sl], tk.k[sl], tk.v[sl], tk.alpha[sl], tk.beta[sl], fold_when_full=False)
        dg = [FoldDiag(128, 128) for _ in range(N)]
        st.fold(diags=dg)
        folds.append(dg)
        for s in range(N):
            S, R = dg[s].S.astype(np.float64), dg[s].R.astype(np.float64)
            sig, lam = st.sigma[s].astype(np.float64), st.lam[s].astype(np.float64)
            step = sig[:, None] * lam[None, :]
            deq = step * st.codes[s].astype(np.float64)
            assert np.all(np.abs(R - deq) <= 0.5 * step * (1 + 1e-4) + 1e-30)
            # compensators copy their lines exactly and leave zeros in the residual
            diff = S - R
            mask = np.zeros_like(S, bool)
            for c in range(4):
                cid = int(st.comp_id[s, c])
                if cid < 128:
                    assert np.array_equal(st.comp_line[s, c], dg[s].S[cid]) or mask[cid].any()
                    mask[cid, :] = True
                else:
                    assert np.array_equal(st.comp_line[s, c], dg[s].S[:, cid - 128]) or mask[:, cid - 128].any()
                    mask[:, cid - 128] = True
            assert np.all(diff[~mask] == 0) and np.all(R[mask] == 0)
            # dequantized boundary plus compensators is within half a step of S
            B = st.dequant(s)
            assert np.all(np.abs(B - S) <= 0.5 * step * (1 + 1e-4) + 1e-30)


# ---------------------------------------------------------------- PIN-5
def test_pin5_planted_lines_are_the_compensators():
    """Two rows and two columns scaled by 30 are the four largest outlier lines."""
    wl = wlm.WORKLOADS[2]
    N = 32
    S0, planted = wlm.initial_state(wl, 0, N)
    st = OracleState(N)
    st.init(S0)
    for s in range(N):
        i1, i2, j1, j2 = (int(x) for x in planted[s])
        assert set(int(c) for c in st.comp_id[s]) == {i1, i2, 128 + j1, 128 + j2}, s


# ---------------------------------------------------------------- PIN-6
@pytest.mark.parametrize("quantize", [False, True])
def test_pin6_associative_memory_closed_form(quantize):
    """alpha = 1, beta = 1, zero start, distinct one-hot keys: the delta rule stores
    v_m under key e_pi(m) exactly (LeapQuant App. A, delta rule)."""
    rng = np.random.default_rng(6)
    T, W = 40, 16
    perm = rng.permutation(128)[:T]
    k = np.zeros((T, 1, 128), np.float32)
    k[np.arange(T), 0, perm] = 1.0
    v = rng.standard_normal((T, 1, 128)).astype(np.float32)
    q = k.copy()
    alpha = np.ones((T, 1), np.float32)
    beta = np.ones((T, 1), np.float32)
    st = OracleState(1, W=W, C=0, smooth=False, quantize=quantize)
    st.init(None)
    steps = []  # sigma after each fold: every fold may move a stored value by half its step
    for t in range(T):
        o = st.run(q[t:t + 1], k[t:t + 1], v[t:t + 1], alpha[t:t + 1], beta[t:t + 1])[0, 0]
        S = st.export()[0]
        if not quantize:
            assert np.array_equal(o.astype(np.float32), v[t, 0])
            for m in range(t + 1):
                assert np.array_equal(S[:, perm[m]], v[m, 0])
        else:
            n_open = (t + 1) % W
            if n_open == 0:
                steps.append(st.sigma[0].astype(np.float64))
            for m in range(t + 1 - n_open, t + 1):  # still exact records
                assert np.array_equal(S[:, perm[m]], v[m, 0])
            for m in range(t + 1 - n_open):  # folded: half a step per fold since it was written
                bound = 0.5 * sum(steps[m // W:]) * (1 + 1e-4) + 1e-30
                assert np.all(np.abs(S[:, perm[m]] - v[m, 0]) <= bound)
                if m // W == len(steps) - 1:
                    assert np.all(np.abs(S[:, perm[m]] - v[m, 0]) <= 0.5 * steps[-1] * (1 + 1e-4) + 1e-30)


# ---------------------------------------------------------------- PIN-7
def test_pin7_beta_zero_fold_is_idempotent():
    wl = wlm.custom(107, 3, 1, n_warm=48)
    S0, _ = wlm.initial_state(wl)
    st = OracleState(3, W=16, C=0, smooth=False)
    st.init(S0)
    codes0, sig0 = st.codes.copy(), st.sigma.copy()
    tk = wlm.tokens(wl, 0, 1)
    ones = np.ones((1, 3), np.float32)
    st.run(tk.q, tk.k, tk.v, ones, 0 * ones, fold_when_full=False)
    st.fold()
    assert np.array_equal(st.codes, codes0)
    assert np.all(np.abs(st.sigma.view(np.int32) - sig0.view(np.int32)) <= 1)


def test_pin7_beta_zero_output_is_boundary_read():
    """beta = 0 (plain gated linear attention, App. A): o_n = B (A_n . q_n)."""
    wl = wlm.WORKLOADS[2]
    S0, _ = wlm.initial_state(wl, 0, 2)
    tk = wlm.tokens(wl, 0, 5, 0, 2)
    st = OracleState(2)
    st.init(S0)
    B = [st.dequant(s) for s in range(2)]
    A = np.ones(2)
    zero = np.zeros_like(tk.beta)
    for t in range(5):
        A = A * tk.alpha[t].astype(np.float64)
        o = st.run(*(x[t:t + 1] for x in (tk.q, tk.k, tk.v, tk.alpha)), zero[t:t + 1], fold_when_full=False)[0]
        for s in range(2):
            ref = B[s] @ (A[s] * tk.q[t, s].astype(np.float64))
            assert rel_l2(o[s], ref) <= 1e-6


# ---------------------------------------------------------------- PIN-9
def test_pin9_power_of_two_scale_invariance():
    """v and S0 times 4: u, S, o and compensator lines times 4; sigma and lambda
    times 2 (4 = 2 * 2); codes and ids unchanged. Powers of two scale exactly."""
    wl = wlm.WORKLOADS[2]
    N, T = 2, 34
    S0, _ = wlm.initial_state(wl, 0, N)
    tk = wlm.tokens(wl, 0, T, 0, N)
    a = OracleState(N)
    b = OracleState(N)
    a.init(S0)
    b.init(4 * S0)
    oa = a.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    ob = b.run(tk.q, tk.k, 4 * tk.v, tk.alpha, tk.beta)
    # The floor is active only on columns taken whole as compensators (zero in the
    # residual, so their scale multiplies zero codes); it does not scale there.
    floored = a.lam == np.float32(1e-6)
    for s, j in zip(*np.nonzero(floored)):
        assert 128 + j in set(int(c) for c in a.comp_id[s])
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.comp_id, b.comp_id)
    assert np.array_equal(2 * a.sigma, b.sigma)
    assert np.array_equal(np.where(floored, a.lam, 2 * a.lam), b.lam)
    assert np.array_equal(4 * a.comp_line, b.comp_line)
    assert np.array_equal(4 * a.rec_u, b.rec_u)
    assert np.array_equal(4 * oa, ob)


# ---------------------------------------------------------------- textbook special cases
@pytest.mark.parametrize("bits", [8, 6, 4])
def test_no_comp_no_smooth_init_is_textbook_per_row_absmax(bits):
    qm = 2 ** (bits - 1) - 1
    rng = np.random.default_rng(11)
    S0 = (rng.standard_normal((4, 128, 128)) * rng.uniform(0.1, 10, (4, 128, 1))).astype(np.float32)
    S0[1, 5, :] = 0.0  # all-zero row: sigma 0, codes 0
    st = OracleState(4, C=0, smooth=False, code_bits=bits)
    st.init(S0)
    f32 = np.float32
    m = np.abs(S0).max(axis=2)
    h = np.where(m > 0, f32(qm) / np.where(m > 0, m, 1), 0).astype(f32)
    ref = np.clip(np.rint((S0 * h[:, :, None]).astype(f32)), -qm, qm).astype(np.int8)
    assert np.array_equal(st.codes, ref)
    assert np.array_equal(st.sigma, np.where(m > 0, m / f32(qm), 0).astype(f32))
    assert (st.codes[1, 5] == 0).all() and st.sigma[1, 5] == 0


def test_smoothing_scales_follow_their_formula():
    """lambda_j = max(sqrt(mean_i |R_ij|), floor) on the residual after compensators
    (LeapQuant §3.4); sigma_i = max_j |R_ij / lambda_j| / 127."""
    wl = wlm.WORKLOADS[5]
    S0, _ = wlm.initial_state(wl, 0, 2)
    S0[1, :, 7] = 0.0  # an all-zero column after selection: the floor applies
    st = OracleState(2, lambda_floor=1e-3)
    dg = [FoldDiag(128, 128) for _ in range(2)]
    st.init(S0, diags=dg)
    for s in range(2):
        R = dg[s].R.astype(np.float64)
        lam = np.maximum(np.sqrt(np.abs(R).mean(axis=0)), 1e-3)
        np.testing.assert_allclose(st.lam[s], lam, rtol=3e-7)
        sig = np.abs(R / st.lam[s].astype(np.float64)[None, :]).max(axis=1) / 127
        np.testing.assert_allclose(st.sigma[s], sig, rtol=5e-7)
    assert st.lam[1, 7] == np.float32(1e-3)


def test_per_window_beats_per_step_rounding():
    """Direction of LeapQuant §3.2 (state error far lower with 16-token windows than
    per-step rounding), on synthetic inputs: a qualitative check only."""
    wl = wlm.custom(120, 4, 256, n_warm=64)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, wl.n_tokens)
    ref = OracleState(4, C=0, quantize=False)
    win = OracleState(4, W=16, C=0, smooth=False)
    step = OracleState(4, W=1, C=0, smooth=False)
    for st in (ref, win, step):
        st.init(S0)
        st.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    e_win = np.linalg.norm(win.export() - ref.export())
    e_step = np.linalg.norm(step.export() - ref.export())
    assert e_win < e_step


def test_window_full_is_an_error():
    st = OracleState(1, W=2, C=0)
    st.init(None)
    x = np.zeros((1, 1, 128), np.float32)
    one = np.ones((1, 1), np.float32)
    st.run(x, x, x, one, one, fold_when_full=False)
    st.run(x, x, x, one, one, fold_when_full=False)
    with pytest.raises(RuntimeError):
        st.run(x, x, x, one, one, fold_when_full=False)


# ---------------------------------------------------------------- F5 at exact ties
@pytest.mark.parametrize("bits", [8, 6, 4])
def test_f5_rounds_exact_ties_to_even(bits):
    """Reading R8 (the pages leave the rounding mode open: research note 4, "Why rounding
    the state is difficult"): F5 rounds half to even. Half away from zero, truncation or
    rounding half up all miss at least one of these typed-out codes."""
    qm = 2 ** (bits - 1) - 1
    S0, want = tie_rows(qm)
    st = OracleState(1, C=0, smooth=False, code_bits=bits)
    dg = [FoldDiag(128, 128)]
    st.init(S0, diags=dg)
    # the values handed to the rounding are the exact half-integers themselves
    assert np.array_equal(dg[0].s_round[:3, :13] * 2, np.rint(dg[0].s_round[:3, :13] * 2))
    assert np.array_equal(st.codes, want)
    assert np.array_equal(st.sigma[0, :3], (np.float32(qm) * np.float32([0.5, 1.0, 2.0])) / np.float32(qm))


# ---------------------------------------------------------------- F2 at exact score ties
@pytest.mark.parametrize("case", range(3))
def test_f2_exact_score_ties_go_to_the_smallest_id(case):
    """Reading R5: among equal squared lengths the smallest id wins, so rows come before
    columns and a smaller column before a larger one; once the residual is zero every score
    ties at 0. Ties to the largest id, columns first or a one-shot top-C all miss one of
    these hand-worked id lists."""
    S0, want = selection_ties()[case]
    st = OracleState(1, W=16, C=4)
    st.init(S0)
    assert st.comp_id[0, :4].tolist() == want
