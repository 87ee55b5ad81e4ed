"""Outputs whose last term nearly cancels, against the exact value.

From a zero state the first token's output is the new record's term alone,
o = u (k . q) with u = beta v (LeapQuant §3.1: the state after one delta-rule
step is beta v k^T). When q is nearly orthogonal to k, k . q is a small
difference of large products and a float32 sum of the 128 products loses most
of its digits. The kernels form that term as a compensated float dot (each
product split into its float value and exact error, the values added with
error-free two-sums and the errors carried beside them): the result is as if
summed in twice the float precision and rounded once, so the output stays
within a few float roundings of the exact value. The
cases cover one-record tokens (scalar and per-key decay), two-record tokens
(q nearly orthogonal to both keys) and RWKV7 tokens (r nearly orthogonal to
the write key; the erase record is empty at a zero state).
"""
import numpy as np
import pytest
import torch

from oracle import OracleState
from quantized_linear_attention_gb300 import lq
from tests._gpu import GpuState, to_dev
from tests._helpers import rel_l2

pytestmark = pytest.mark.gpu

EPS = 1e-6  # |k . q| / (|k| |q|) before rounding q to float32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _near_orthogonal(rng, keys):
    """Queries with |q| ~ 1 orthogonal to every key in `keys` up to EPS along the first."""
    q = rng.standard_normal(keys[0].shape)
    basis = []
    for k in keys:
        b = k.astype(np.float64)
        for e in basis:
            b = b - np.sum(b * e, axis=1, keepdims=True) * e
        basis.append(_unit(b))
    for e in basis:
        q = q - np.sum(q * e, axis=1, keepdims=True) * e
    q = _unit(q) + EPS * basis[0]
    return q.astype(np.float32)


def _token(rng, n, kda):
    k = _unit(rng.standard_normal((n, 128))).astype(np.float32)
    v = rng.standard_normal((n, 128)).astype(np.float32)
    a = rng.uniform(0.9, 1.0, (n, 128) if kda else (n,)).astype(np.float32)
    b = rng.uniform(0.2, 1.0, n).astype(np.float32)
    return k, v, a, b


@pytest.mark.parametrize("kda", [False, True])
def test_first_token_from_zero_state_is_exact(kda):
    rng = np.random.default_rng(1500 + kda)
    n = 300
    k, v, a, b = _token(rng, n, kda)
    q = _near_orthogonal(rng, [k])
    kq = np.sum(k.astype(np.float64) * q.astype(np.float64), axis=1)
    assert np.all(np.abs(kq) < 1e-5)  # the cancellation the case is about
    gpu = GpuState(n, W=16, C=4, kda=kda)
    gpu.init(None)
    o = gpu.step(*(to_dev(x) for x in (q, k, v, a, b)), phase=0).cpu().numpy()
    u = (b[:, None] * v).astype(np.float32)  # u = beta (v - S_0 k) rounded, S_0 = 0
    exact = u.astype(np.float64) * kq[:, None]
    assert rel_l2(o, exact).max() <= 1e-6
    ref = OracleState(n, W=16, C=4, decay_per_key=kda)
    ref.init(None)
    o_ref = ref.run(q[None], k[None], v[None], a[None], b[None])[0]
    assert rel_l2(o, o_ref).max() <= 1e-6
    assert gpu.status()[0] == lq.OK


def test_two_record_token_from_zero_state():
    rng = np.random.default_rng(1510)
    n = 200
    k1, v1, a, b1 = _token(rng, n, False)
    k2, v2, _, b2 = _token(rng, n, False)
    q = _near_orthogonal(rng, [k1, k2])
    gpu = GpuState(n, W=16, C=4)
    gpu.init(None)
    lq.decode_step2(gpu.cfg, gpu.state, n, *(to_dev(x) for x in (q, k1, v1, b1, k2, v2, b2, a)), gpu.o, phase=0)
    ref = OracleState(n, W=16, C=4)
    ref.init(None)
    ref.run(q[None], k1[None], v1[None], a[None], b1[None], fold_when_full=False)
    o_ref = ref.run(q[None], k2[None], v2[None], np.ones_like(a)[None], b2[None], fold_when_full=False)[0]
    assert rel_l2(gpu.o.cpu().numpy(), o_ref).max() <= 1e-5
    assert gpu.status()[0] == lq.OK


def test_rwkv7_token_from_zero_state():
    rng = np.random.default_rng(1520)
    n = 200
    k1, _, a, _ = _token(rng, n, True)
    k, v, ka, _ = _token(rng, n, True)
    kh = _unit(k1.astype(np.float64)).astype(np.float32)
    r = _near_orthogonal(rng, [k])
    gpu = GpuState(n, W=16, C=4, kda=True)
    gpu.init(None)
    lq.decode_step_rwkv7(gpu.cfg, gpu.state, n, *(to_dev(x) for x in (r, a, kh, ka, k, v)), gpu.o, phase=0)
    ref = OracleState(n, W=16, C=4, decay_per_key=True)
    ref.init(None)
    o_ref = ref.append_rwkv(r, a, kh, ka, k, v)
    assert rel_l2(gpu.o.cpu().numpy(), o_ref).max() <= 1e-6
    assert gpu.status()[0] == lq.OK
