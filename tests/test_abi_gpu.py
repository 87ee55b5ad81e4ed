"""Device-side status and host-side validation of the C ABI on a GPU (no fault is provoked:
every bad argument is caught on the host, every bad state on the device by a check)."""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(n, t=0, kda=False):
    wl = wlm.custom(500, n, 0, kda=kda)
    tk = wlm.tokens(wl, t, 1)
    return [torch.from_numpy(np.ascontiguousarray(x[0])).to(DEV) for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta)]


def _fresh(n=4, **kw):
    cfg = lq.config(**kw)
    st = lq.alloc_state(cfg, n, DEV)
    lq.state_init(cfg, st, n, None)
    return cfg, st


def test_window_full_sets_status_and_leaves_state():
    cfg, st = _fresh(4, window=3)
    q, k, v, a, b = _inputs(4)
    o = torch.empty(4, 128, device=DEV)
    for _ in range(3):
        lq.append(cfg, st, 4, q, k, v, a, b, o)
    assert lq.get_status(st)[0] == lq.OK
    before = st.clone()
    lq.append(cfg, st, 4, q, k, v, a, b, o)
    status, bad = lq.get_status(st)
    assert status == lq.ERR_WINDOW_FULL and 0 <= bad < 4
    lay = lq.layout(cfg, 4)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    lq.clear_status(st)
    assert lq.get_status(st) == (lq.OK, -1)
    lq.fold(cfg, st, 4)
    lq.append(cfg, st, 4, q, k, v, a, b, o)
    assert lq.get_status(st)[0] == lq.OK


def test_phase_mismatch_sets_status_and_leaves_state():
    cfg, st = _fresh(5)
    q, k, v, a, b = _inputs(5)
    o = torch.zeros(5, 128, device=DEV)
    before = st.clone()
    lq.decode_step(cfg, st, 5, q, k, v, a, b, o, phase=3)
    assert lq.get_status(st)[0] == lq.ERR_PHASE
    lay = lq.layout(cfg, 5)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    assert float(o.abs().sum()) == 0.0
    lq.clear_status(st)
    lq.decode_step(cfg, st, 5, q, k, v, a, b, o, phase=15)  # fused kernel path, still the wrong phase
    assert lq.get_status(st)[0] == lq.ERR_PHASE


def test_uninitialised_or_foreign_state_is_rejected_on_device():
    cfg = lq.config()
    n = 3
    st = torch.zeros(lq.state_bytes(cfg, n), dtype=torch.uint8, device=DEV)
    q, k, v, a, b = _inputs(n)
    o = torch.empty(n, 128, device=DEV)
    lq.decode_step(cfg, st, n, q, k, v, a, b, o)
    assert lq.get_status(st)[0] == lq.ERR_STATE  # magic missing
    # initialised with another configuration: the header hash differs
    cfg_a = lq.config(window=8)
    lq.state_init(cfg_a, st, n, None)
    assert lq.get_status(st)[0] == lq.OK
    lq.fold(lq.config(window=8, n_comp=3), st, n)
    assert lq.get_status(st)[0] == lq.ERR_STATE


def test_host_validation_launches_nothing():
    cfg, st = _fresh(4)
    q, k, v, a, b = _inputs(4)
    o = torch.empty(4, 128, device=DEV)
    with pytest.raises(lq.LQError) as e:
        lq.append(cfg, st, 4, 0, k, v, a, b, o)
    assert e.value.code == lq.ERR_INVALID_ARG
    with pytest.raises(lq.LQError) as e:  # misaligned input
        lq.append(cfg, st, 4, q.data_ptr() + 4, k, v, a, b, o)
    assert e.value.code == lq.ERR_INVALID_ARG
    host = torch.zeros(4, 128).pin_memory()
    with pytest.raises(lq.LQError) as e:  # pinned host memory is not device memory
        lq.append(cfg, st, 4, host.data_ptr(), k, v, a, b, o)
    assert e.value.code == lq.ERR_INVALID_ARG
    with pytest.raises(lq.LQError) as e:  # o aliases q
        lq.append(cfg, st, 4, q, k, v, a, b, q)
    assert e.value.code == lq.ERR_INVALID_ARG
    with pytest.raises(lq.LQError) as e:
        lq.decode_step(cfg, st, 4, q, k, v, a, b, o, phase=16)
    assert e.value.code == lq.ERR_INVALID_ARG
    with pytest.raises(lq.LQError) as e:  # state not 256-byte aligned
        lq.fold(cfg, st.data_ptr() + 16, 4)
    assert e.value.code == lq.ERR_INVALID_ARG
    lay = lq.layout(cfg, 4)
    counts = st[lay.counts:lay.counts + 16].view(torch.int32)
    assert counts.tolist() == [0, 0, 0, 0]
    assert lq.get_status(st)[0] == lq.OK


def test_zero_states_is_a_no_op():
    cfg, st = _fresh(1)
    lq.decode_step(cfg, st, 0, 0, 0, 0, 0, 0, 0)
    lq.fold(cfg, st, 0)
    assert lq.get_status(st)[0] == lq.OK


def test_export_mid_window_equals_oracle():
    from oracle import OracleState

    wl = wlm.custom(510, 7, 0, n_warm=40, plant=True)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, 9)
    cfg = lq.config()
    st = lq.alloc_state(cfg, 7, DEV)
    lq.state_init(cfg, st, 7, torch.from_numpy(S0).to(DEV))
    o = torch.empty(7, 128, device=DEV)
    for t in range(9):
        q, k, v, a, b = (torch.from_numpy(np.ascontiguousarray(x)).to(DEV) for x in tk.token(t))
        lq.decode_step(cfg, st, 7, q, k, v, a, b, o, phase=t)
    out = torch.empty(7, 128, 128, device=DEV)
    lq.export_state(cfg, st, 7, out)
    ref = OracleState(7)
    ref.init(S0)
    ref.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta)
    assert np.array_equal(out.cpu().numpy(), ref.export())
