"""The fp32-state baseline kernel (lq_fp32_decode_step) against the oracle's
double-precision recurrence. Its summation order is not pinned, so outputs and
states are compared per head-state by relative L2 error: fp32 rounding over a
few dozen tokens stays near 1e-6, and 1e-5 is the bound."""
import numpy as np
import pytest
import torch

from oracle import fp32_run
from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._helpers import rel_l2

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _run_gpu(cfg, S0, tk, T):
    n = S0.shape[0]
    S = _dev(S0.astype(np.float32))
    o = torch.empty((n, 128), dtype=torch.float32, device=DEV)
    outs = []
    for t in range(T):
        q, k, v, a, b = (_dev(x) for x in tk.token(t))
        lq.fp32_decode_step(cfg, S, n, q, k, v, a, b, o)
        outs.append(o.cpu().numpy().copy())
    return S.cpu().numpy(), np.stack(outs)


@pytest.mark.parametrize("kda", [False, True])
def test_fp32_step_matches_recurrence(kda):
    wl = wlm.custom(520 + int(kda), 7, 0, kda=kda, vdist="t3" if kda else "normal", n_warm=40, plant=not kda)
    S0, _ = wlm.initial_state(wl)
    T = 24
    tk = wlm.tokens(wl, 0, T)
    cfg = lq.config(kda=kda)
    S_g, o_g = _run_gpu(cfg, S0, tk, T)
    S_r, o_r = fp32_run(S0, tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    assert rel_l2(o_g.reshape(-1, 128), o_r.reshape(-1, 128)).max() <= TOL
    assert rel_l2(S_g.reshape(7, -1), S_r.reshape(7, -1)).max() <= TOL


def test_fp32_step_full_batch_sampled():
    """All 16,384 head-states of the batch-512 layer for 4 tokens; the oracle follows a sample."""
    wl = wlm.WORKLOADS[4]
    S0, _ = wlm.initial_state(wl)
    T = 4
    tk = wlm.tokens(wl, 0, T)
    cfg = lq.config()
    S_g, o_g = _run_gpu(cfg, S0, tk, T)
    sample = [0, 1, 777, 8191, 12000, wl.n_states - 1]
    sub = tk.select_states(sample)
    S_r, o_r = fp32_run(S0[sample], sub.q, sub.k, sub.v, sub.alpha, sub.beta)
    assert rel_l2(o_g[:, sample].reshape(-1, 128), o_r.reshape(-1, 128)).max() <= TOL
    assert rel_l2(S_g[sample].reshape(len(sample), -1), S_r.reshape(len(sample), -1)).max() <= TOL


def test_fp32_step_argument_errors():
    cfg = lq.config()
    S = torch.zeros((2, 128, 128), dtype=torch.float32, device=DEV)
    x = torch.zeros((2, 128), dtype=torch.float32, device=DEV)
    s2 = torch.zeros(2, dtype=torch.float32, device=DEV)
    lq.fp32_decode_step(cfg, S, 0, x, x, x, s2, s2, x)  # no head-states: nothing to do
    with pytest.raises(lq.LQError) as e:
        lq.fp32_decode_step(cfg, S.view(-1)[1:], 1, x, x, x, s2, s2, x[1])  # S not 16-byte aligned
    assert e.value.code == lq.ERR_INVALID_ARG
    with pytest.raises(lq.LQError) as e:
        lq.fp32_decode_step(cfg, S, 2, x, x, x, s2, s2, S.view(-1)[:256].view(2, 128))  # o inside S
    assert e.value.code == lq.ERR_INVALID_ARG
