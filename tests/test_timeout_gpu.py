"""Every bounded wait in the kernels, made to run out (no GPU fault is provoked).

The test hook lq_debug_set_wait shortens this thread's bound on the kernels' waits
to 1 ms and makes the append or the fold kernels announce 16 bytes more to their
barrier than they copy: every real copy lands, the barrier never completes, and the
wait gives up. The kernel must then record LQ_ERR_TIMEOUT with the index of a
head-state it was given, write nothing, and return, so that the context stays
usable: a later call with the hook off runs normally. lq_state_init has no such
wait (it reads S0 with plain loads), so it has no case here.
"""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
N, W = 5, 4
WAIT_NS = 1_000_000


@pytest.fixture(autouse=True)
def _hook_off():
    lq.load()
    torch.cuda.set_device(DEV)
    lq.debug_set_wait(0, 0, 0)
    yield
    lq.debug_set_wait(0, 0, 0)


def _setup(kda=False, records=0, phase_any=False):
    wl = wlm.custom(820 + kda, N, 0, kda=kda, n_warm=16, plant=True)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, 2 * W)
    cfg = lq.config(window=W, n_comp=2, kda=kda)
    st = lq.alloc_state(cfg, N, DEV)
    lq.state_init(cfg, st, N, to_dev(S0))
    o = torch.empty((N, 128), dtype=torch.float32, device=DEV)
    for t in range(records):
        lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(t)), o, phase=lq.PHASE_ANY if phase_any else t)
    assert lq.get_status(st) == (lq.OK, -1)
    return cfg, st, tk, o


def _timed_out(st):
    status, bad = lq.get_status(st)
    assert status == lq.ERR_TIMEOUT, lq.STATUS_NAMES.get(status)
    assert 0 <= bad < N


def _usable_again(cfg, st, tk, o):
    """With the hook off, a re-initialised state decodes a token cleanly."""
    lq.debug_set_wait(0, 0, 0)
    lq.state_init(cfg, st, N, None)
    lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(0)), o, phase=0)
    assert lq.get_status(st) == (lq.OK, -1)


@pytest.mark.parametrize("kda", [False, True])
def test_append_wait_runs_out(kda):
    cfg, st, tk, o = _setup(kda, records=1)
    before = st.clone()
    o.fill_(7.0)
    lq.debug_set_wait(WAIT_NS, 16, 0)
    lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(1)), o, phase=1)
    _timed_out(st)
    lay = lq.layout(cfg, N)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    assert bool((o == 7.0).all())
    _usable_again(cfg, st, tk, o)


def test_two_record_wait_runs_out():
    cfg, st, tk, o = _setup(False)
    before = st.clone()
    lq.debug_set_wait(WAIT_NS, 16, 0)
    q, k1, v1, a, b1 = (to_dev(x) for x in tk.token(0))
    _, k2, v2, _, b2 = (to_dev(x) for x in tk.token(1))
    lq.decode_step2(cfg, st, N, q, k1, v1, b1, k2, v2, b2, a, o, phase=0)
    _timed_out(st)
    lay = lq.layout(cfg, N)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    _usable_again(cfg, st, tk, o)


def test_rwkv7_wait_runs_out():
    cfg, st, tk, o = _setup(True)
    before = st.clone()
    lq.debug_set_wait(WAIT_NS, 16, 0)
    r, w, k, v = (to_dev(x) for x in (tk.q[0], tk.alpha[0], tk.k[1], tk.v[1]))
    kh = to_dev(tk.k[0])
    a = to_dev(tk.alpha[1])
    lq.decode_step_rwkv7(cfg, st, N, r, w, kh, a, k, v, o, phase=0)
    _timed_out(st)
    lay = lq.layout(cfg, N)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    _usable_again(cfg, st, tk, o)


@pytest.mark.parametrize("kda", [False, True])
def test_fused_fold_step_wait_runs_out(kda):
    cfg, st, tk, o = _setup(kda, records=W - 1)
    before = st.clone()
    lq.debug_set_wait(WAIT_NS, 0, 16)
    lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(W - 1)), o, phase=W - 1)
    _timed_out(st)
    lay = lq.layout(cfg, N)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    _usable_again(cfg, st, tk, o)


def test_fold_wait_runs_out():
    cfg, st, tk, o = _setup(False, records=2)
    before = st.clone()
    lq.debug_set_wait(WAIT_NS, 0, 16)
    lq.fold(cfg, st, N)
    _timed_out(st)
    lay = lq.layout(cfg, N)
    assert torch.equal(st[lay.counts:], before[lay.counts:])
    _usable_again(cfg, st, tk, o)


@pytest.mark.parametrize("kda", [False, True])
def test_list_fold_wait_runs_out(kda):
    """The mixed-phase step's append fills every window and lists it; the list fold's
    wait runs out, so the windows stay full and unfolded and the list is emptied."""
    cfg, st, tk, o = _setup(kda, records=W - 1, phase_any=True)
    views = lq.state_views(cfg, st, N)
    codes0 = views["codes"].clone()
    lq.debug_set_wait(WAIT_NS, 0, 16)
    lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(W - 1)), o)
    _timed_out(st)
    assert bool((views["counts"] == W).all())
    assert torch.equal(views["codes"], codes0)
    hdr = st[:256].view(torch.int32).cpu().numpy()
    assert hdr[10] == 0 and hdr[11] == 0  # list length and list-fold CTAs done, reset
    _usable_again(cfg, st, tk, o)


def test_export_wait_runs_out():
    cfg, st, tk, o = _setup(False, records=2)
    out = torch.full((N, 128, 128), 3.0, dtype=torch.float32, device=DEV)
    lq.debug_set_wait(WAIT_NS, 0, 16)
    lq.export_state(cfg, st, N, out)
    _timed_out(st)
    assert bool((out == 3.0).all())
    _usable_again(cfg, st, tk, o)

