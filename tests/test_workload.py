"""The seeded synthetic input generator (no GPU)."""
import numpy as np

from quantized_linear_attention_gb300 import workload as wlm


def test_splitmix64_published_first_outputs():
    # SplitMix64 from seed 0 (Steele, Lea, Flood 2014): the first two outputs are
    # mix64(gamma) and mix64(2 * gamma).
    g = 0x9E3779B97F4A7C15
    assert wlm.mix64(g) == 0xE220A8397B1DCDAF
    assert wlm.mix64((2 * g) % 2**64) == 0x6E789E6AA1B965F4


def test_distributions():
    wl = wlm.WORKLOADS[2]
    tk = wlm.tokens(wl, 0, 8, 0, 256)
    np.testing.assert_allclose(np.linalg.norm(tk.q, axis=-1), 1.0, rtol=1e-6)
    np.testing.assert_allclose(np.linalg.norm(tk.k, axis=-1), 1.0, rtol=1e-6)
    assert abs(tk.v.mean()) < 0.02 and abs(tk.v.std() - 1) < 0.02
    assert tk.alpha.min() == np.float32(0.8) and tk.alpha.max() < 1.0
    # alpha = 1/(1+e^x) >= 0.8 iff x <= ln(1/4): P = Phi(-1.386) = 0.083
    assert abs((tk.alpha > np.float32(0.8)).mean() - 0.083) < 0.02
    assert 0 < tk.beta.min() and tk.beta.max() < 1 and abs(tk.beta.mean() - 0.5) < 0.02


def test_kda_distributions():
    wl = wlm.WORKLOADS[5]
    tk = wlm.tokens(wl, 0, 2, 0, 64)
    assert tk.alpha.shape == (2, 64, 128)
    assert abs(np.median(tk.alpha) - 0.5) < 0.02
    # Student-t(3): variance 3, heavy tails
    assert abs(tk.v.var() - 3.0) < 0.6 and np.abs(tk.v).max() > 8


def test_subsets_regenerate_the_same_values():
    wl = wlm.WORKLOADS[3]
    full = wlm.tokens(wl, 10, 4, 0, 16)
    sub = wlm.tokens(wl, 11, 2, states=[3, 9, 15])
    assert np.array_equal(sub.q, full.q[1:3, [3, 9, 15]])
    assert np.array_equal(sub.v, full.v[1:3, [3, 9, 15]])
    assert np.array_equal(sub.beta, full.beta[1:3, [3, 9, 15]])
    a = wlm.tokens(wl, 0, 1, 5, 3, nthreads=1)
    b = wlm.tokens(wl, 0, 1, 5, 3, nthreads=3)
    assert np.array_equal(a.k, b.k)


def test_initial_state_planting():
    wl = wlm.WORKLOADS[2]
    S0, planted = wlm.initial_state(wl, 0, 8)
    for s in range(8):
        i1, i2, j1, j2 = planted[s]
        assert i1 != i2 and j1 != j2
        rn = np.linalg.norm(S0[s], axis=1)
        cn = np.linalg.norm(S0[s], axis=0)
        assert set(np.argsort(rn)[-2:]) == {i1, i2}
        assert set(np.argsort(cn)[-2:]) == {j1, j2}
    S0b, _ = wlm.initial_state(wl, states=[5])
    assert np.array_equal(S0b[0], S0[5])
    assert wlm.initial_state(wlm.WORKLOADS[1])[0] is None


def test_workload_shapes_match_pages():
    from tests._helpers import read_golden

    g = read_golden("page_figures.txt")
    w4 = wlm.WORKLOADS[4]
    assert w4.heads == g["qwen35_9b_heads"] and w4.dk == w4.dv == g["state_rows"] and w4.W == g["window_tokens"]
    assert wlm.WORKLOADS[2].n_tokens == g["trace_tokens"]
    w5 = wlm.WORKLOADS[5]
    assert w5.layers == g["qwen35_9b_linear_layers"]
    per_request = g["qwen35_9b_linear_layers"] * g["qwen35_9b_heads"] * g["state_rows"] ** 2 * 4
    assert round(per_request / 1e6, 1) == g["qwen35_9b_fp32_state_mb"]
    # one verified trace: its 510 folds covered 32 heads of 128 x 128 entries each
    assert g["verified_entries"] == g["verified_folds"] * g["qwen35_9b_heads"] * g["state_rows"] ** 2
