"""Pin: a two-record token in the oracle is the DeltaProduct update with two steps.

LeapQuant App. A ("Instances of the general update") writes a token whose
update takes two rank-one sub-steps as two records; for a DeltaProduct token
with two steps the first record carries the token's decay and the second
decay 1. With quantization off, two oracle appends per token must follow the
product form of that recurrence, computed here in float64 with explicit
matrices (a different expression from the records' sum):
    S_t = S_{t-1} D (I - b1 k1 k1^T)(I - b2 k2 k2^T) + b1 v1 k1^T (I - b2 k2 k2^T) + b2 v2 k2^T,
    o_t = S_t q_t.
Putting the decay on the second record, swapping the sub-steps or reading the
second sub-step from S_{t-1} each moves the result far outside the bound.
"""
import numpy as np
import pytest

from oracle import OracleState


def _tokens(rng, T, n, kda):
    def unit(x):
        return x / np.linalg.norm(x, axis=-1, keepdims=True)

    k1 = unit(rng.standard_normal((T, n, 128))).astype(np.float32)
    k2 = unit(rng.standard_normal((T, n, 128))).astype(np.float32)
    q = (rng.standard_normal((T, n, 128)) / np.sqrt(128)).astype(np.float32)
    v1 = rng.standard_normal((T, n, 128)).astype(np.float32)
    v2 = rng.standard_normal((T, n, 128)).astype(np.float32)
    b1 = rng.uniform(0.1, 0.9, (T, n)).astype(np.float32)
    b2 = rng.uniform(0.1, 0.9, (T, n)).astype(np.float32)
    a = rng.uniform(0.9, 1.0, (T, n, 128) if kda else (T, n)).astype(np.float32)
    return q, k1, v1, b1, k2, v2, b2, a


def _product_form(S, q, k1, v1, b1, k2, v2, b2, a, kda):
    I = np.eye(128)
    D = np.diag(a.astype(np.float64)) if kda else float(a) * I
    H1 = I - float(b1) * np.outer(k1, k1)
    H2 = I - float(b2) * np.outer(k2, k2)
    S = S @ D @ H1 @ H2 + float(b1) * np.outer(v1, k1) @ H2 + float(b2) * np.outer(v2, k2)
    return S, S @ q.astype(np.float64)


@pytest.mark.parametrize("kda", [False, True])
def test_two_records_per_token_follow_the_product_form(kda):
    rng = np.random.default_rng(41 + kda)
    n, T, W = 3, 13, 8  # 13 tokens: three folds (every four tokens), then a part window
    q, k1, v1, b1, k2, v2, b2, a = _tokens(rng, T, n, kda)
    S0 = rng.standard_normal((n, 128, 128)).astype(np.float32) * 0.1
    ref = OracleState(n, W=W, C=0, decay_per_key=kda, quantize=False)
    ref.init(S0)
    ones = np.ones_like(a[0])
    S = S0.astype(np.float64)
    worst_o = worst_s = 0.0
    for t in range(T):
        ref.run(q[t][None], k1[t][None], v1[t][None], a[t][None], b1[t][None], fold_when_full=True)
        o = ref.run(q[t][None], k2[t][None], v2[t][None], ones[None], b2[t][None], fold_when_full=True)[0]
        for s in range(n):
            S[s], o_ref = _product_form(S[s], q[t, s], k1[t, s], v1[t, s], b1[t, s], k2[t, s], v2[t, s], b2[t, s],
                                        a[t, s], kda)
            worst_o = max(worst_o, np.linalg.norm(o[s] - o_ref) / np.linalg.norm(o_ref))
        ex = ref.export().astype(np.float64)
        worst_s = max(worst_s, np.linalg.norm(ex - S) / np.linalg.norm(S))
    assert worst_o < 2e-5 and worst_s < 2e-5, (worst_o, worst_s)


def test_the_product_form_rejects_a_decayed_second_record():
    """The same check catches the plausible mistake of decaying the second record too."""
    rng = np.random.default_rng(7)
    q, k1, v1, b1, k2, v2, b2, a = _tokens(rng, 4, 1, False)
    a[:] = 0.5  # a strong decay makes the difference large
    S0 = rng.standard_normal((1, 128, 128)).astype(np.float32) * 0.1
    ref = OracleState(1, W=8, C=0, quantize=False)
    ref.init(S0)
    S = S0[0].astype(np.float64)
    for t in range(4):
        ref.run(q[t][None], k1[t][None], v1[t][None], a[t][None], b1[t][None])
        o = ref.run(q[t][None], k2[t][None], v2[t][None], a[t][None], b2[t][None])[0]  # wrong: decays twice
        S, o_ref = _product_form(S, q[t, 0], k1[t, 0], v1[t, 0], b1[t, 0], k2[t, 0], v2[t, 0], b2[t, 0], a[t, 0],
                                 False)
    assert np.linalg.norm(o[0] - o_ref) / np.linalg.norm(o_ref) > 1e-2
