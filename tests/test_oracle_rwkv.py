"""Pin: an RWKV7 token in the oracle is two records that follow RWKV7's update.

LeapQuant App. A ("Instances of the general update") represents RWKV7, whose
erase direction differs from its write key, by an erase sub-step and a
pure-write sub-step: two rank-one records per token. With quantization off,
the oracle's records must follow the update written as a matrix product,
computed here in float64:
    S_t = S_{t-1} (Diag(w) - kh (a . kh)^T) + v k^T,    o_t = S_t r.
Reading the erase from the decayed state, or writing it along kh instead of
a . kh, moves the result far outside the bound (checked below).
"""
import numpy as np

from oracle import OracleState


def _tokens(rng, T, n):
    def unit(x):
        return x / np.linalg.norm(x, axis=-1, keepdims=True)

    r = (rng.standard_normal((T, n, 128)) / np.sqrt(128)).astype(np.float32)
    w = rng.uniform(0.85, 1.0, (T, n, 128)).astype(np.float32)
    kh = unit(rng.standard_normal((T, n, 128))).astype(np.float32)
    a = rng.uniform(0.2, 1.0, (T, n, 128)).astype(np.float32)
    k = (rng.standard_normal((T, n, 128)) / np.sqrt(128)).astype(np.float32)
    v = rng.standard_normal((T, n, 128)).astype(np.float32)
    return r, w, kh, a, k, v


def _step(S, r, w, kh, a, k, v):
    kh64, a64 = kh.astype(np.float64), a.astype(np.float64)
    M = np.diag(w.astype(np.float64)) - np.outer(kh64, (a64 * kh64).astype(np.float32).astype(np.float64))
    S = S @ M + np.outer(v, k)
    return S, S @ r.astype(np.float64)


def test_rwkv_tokens_follow_the_rwkv7_update_across_folds():
    rng = np.random.default_rng(51)
    n, T, W = 3, 11, 6  # three records... two per token: a fold every three tokens
    r, w, kh, a, k, v = _tokens(rng, T, n)
    S0 = (rng.standard_normal((n, 128, 128)) * 0.05).astype(np.float32)
    ref = OracleState(n, W=W, C=0, decay_per_key=True, quantize=False)
    ref.init(S0)
    S = S0.astype(np.float64)
    worst_o = worst_s = 0.0
    for t in range(T):
        o = ref.append_rwkv(r[t], w[t], kh[t], a[t], k[t], v[t])
        for s in range(n):
            S[s], o_ref = _step(S[s], r[t, s], w[t, s], kh[t, s], a[t, s], k[t, s], v[t, s])
            worst_o = max(worst_o, np.linalg.norm(o[s] - o_ref) / np.linalg.norm(o_ref))
        if ref.count[0] == W:
            ref.fold()
        worst_s = max(worst_s, np.linalg.norm(ref.export() - S) / np.linalg.norm(S))
    assert worst_o < 2e-5 and worst_s < 2e-5, (worst_o, worst_s)


def test_the_erase_reads_the_state_before_the_decay():
    """The same check rejects an erase that reads the decayed state S Diag(w) kh."""
    rng = np.random.default_rng(52)
    r, w, kh, a, k, v = _tokens(rng, 3, 1)
    w[:] = 0.5
    S0 = (rng.standard_normal((1, 128, 128)) * 0.05).astype(np.float32)
    ref = OracleState(1, W=8, C=0, decay_per_key=True, quantize=False)
    ref.init(S0)
    S = S0[0].astype(np.float64)
    for t in range(3):
        o = ref.append_rwkv(r[t], w[t], kh[t], a[t], k[t], v[t])[0]
        M = np.diag(w[t, 0].astype(np.float64))
        wrong = S @ M - np.outer(S @ M @ kh[t, 0], a[t, 0] * kh[t, 0]) + np.outer(v[t, 0], k[t, 0])
        S, o_ref = _step(S, r[t, 0], w[t, 0], kh[t, 0], a[t, 0], k[t, 0], v[t, 0])
    assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) < 2e-5
    o_wrong = wrong @ r[2, 0].astype(np.float64)
    assert np.linalg.norm(o_wrong - o_ref) / np.linalg.norm(o_ref) > 1e-2


def test_rwkv_records_are_the_erase_then_the_pure_write():
    rng = np.random.default_rng(53)
    r, w, kh, a, k, v = _tokens(rng, 1, 2)
    ref = OracleState(2, W=4, C=2, decay_per_key=True)
    ref.init(None)
    ref.append_rwkv(r[0], w[0], kh[0], a[0], k[0], v[0])
    assert ref.count.tolist() == [2, 2]
    assert np.array_equal(ref.rec_k[:, 0], a[0] * kh[0])
    assert np.array_equal(ref.rec_alpha[:, 0], w[0]) and np.array_equal(ref.rec_alpha[:, 1], np.ones_like(w[0]))
    assert np.array_equal(ref.rec_k[:, 1], k[0]) and np.array_equal(ref.rec_u[:, 1], v[0])
    assert not ref.rec_u[:, 0].any()  # a zero state: the erase removes nothing
