"""Pins of the oracle's fp32-state baseline recurrence (the plain per-token delta
rule on a whole state; LeapQuant §3.1 and App. A), against results it does not
compute itself."""
import numpy as np
import pytest

from oracle import OracleState, fp32_run
from quantized_linear_attention_gb300 import workload as wlm
from tests._helpers import rel_l2


@pytest.mark.parametrize("wid,N,T", [(2, 3, 40), (5, 2, 40)])
def test_fp32_recurrence_equals_windowed_unquantized_form(wid, N, T):
    """The window unrolling (records, decay products, fold without rounding) and
    the per-token recurrence are two computations of the same states (App. B.2)."""
    wl = wlm.WORKLOADS[wid]
    S0, _ = wlm.initial_state(wl, 0, N)
    tk = wlm.tokens(wl, 0, T, 0, N)
    st = OracleState(N, W=16, C=0, decay_per_key=wl.kda, quantize=False)
    st.init(S0)
    o_win = st.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    S_T, o = fp32_run(S0, tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    assert rel_l2(o.reshape(-1, 128), o_win.reshape(-1, 128)).max() <= 1e-5
    assert rel_l2(S_T.reshape(N, -1), st.export().reshape(N, -1)).max() <= 1e-5


def test_fp32_recurrence_associative_memory_exact():
    """alpha = beta = 1, zero start, distinct one-hot keys: the state stores v_m
    under key e_pi(m) exactly and o_t = v_t for q_t = k_t (delta rule, App. A)."""
    rng = np.random.default_rng(10)
    T = 50
    perm = rng.permutation(128)[:T]
    k = np.zeros((T, 1, 128), np.float32)
    k[np.arange(T), 0, perm] = 1.0
    v = rng.standard_normal((T, 1, 128)).astype(np.float32)
    S, o = fp32_run(np.zeros((1, 128, 128)), k, k, v, np.ones((T, 1), np.float32), np.ones((T, 1), np.float32))
    assert np.array_equal(o[:, 0], v[:, 0].astype(np.float64))
    for m in range(T):
        assert np.array_equal(S[0][:, perm[m]], v[m, 0].astype(np.float64))
    rest = np.setdiff1d(np.arange(128), perm)
    assert not S[0][:, rest].any()


def test_fp32_recurrence_beta_zero_is_pure_decay():
    """beta = 0: no write, so S_T = S_0 times the product of the decays (KDA: per key column)."""
    wl = wlm.WORKLOADS[5]
    S0, _ = wlm.initial_state(wl, 0, 2)
    tk = wlm.tokens(wl, 0, 12, 0, 2)
    beta = np.zeros_like(tk.beta)
    S_T, _ = fp32_run(S0, tk.q, tk.k, tk.v, tk.alpha, beta, want_o=False)
    decay = np.prod(tk.alpha.astype(np.float64), axis=0)  # [n][d_k]
    expect = S0.astype(np.float64) * decay[:, None, :]
    assert np.allclose(S_T, expect, rtol=1e-14, atol=0)
