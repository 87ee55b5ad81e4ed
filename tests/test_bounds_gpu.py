"""Guard words around every buffer, in place of a memory checker (compute-sanitizer is
closed on this pool).

Every buffer a call touches sits inside a larger allocation whose guard regions (4 KB
before and after) hold a byte pattern, and the state buffer itself is filled with the
pattern before it is initialised. Ragged head-state counts run through every call of
the C ABI: stated-phase decode steps (append-only and the fused last token), mixed-phase
steps with the list fold, a range re-initialisation, lq_fold, two-record or RWKV7
tokens and lq_export_state. After each call:
  - every guard still holds the pattern and no input changed;
  - inside the state buffer, the bytes that changed all lie where that call's work
    lands: the record counts, the record slot each head-state filled, the boundaries
    of the head-states that folded or were initialised, the work list, and the header
    fields the whole-buffer init writes. Padding between planes, the record slots
    beyond each window's fill and every other head-state's slice are untouched.
"""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096
PAT = 0xA5


class Guarded:
    """nbytes inside a pattern-filled allocation with GUARD bytes on each side."""

    def __init__(self, nbytes, data=None):
        self.n = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), PAT, dtype=torch.uint8, device=DEV)
        self.inner = self.raw[GUARD:GUARD + nbytes]
        if data is not None:
            self.inner.copy_(torch.from_numpy(np.ascontiguousarray(data)).view(-1).view(torch.uint8).to(DEV))
        self.snap = self.inner.clone()

    def f32(self):
        return self.inner.view(torch.float32)

    def guards_ok(self):
        return bool((self.raw[:GUARD] == PAT).all()) and bool((self.raw[GUARD + self.n:] == PAT).all())


class Regions:
    """Byte ranges of a state buffer a call may write."""

    def __init__(self, cfg, n):
        self.cfg, self.n, self.L = cfg, n, lq.layout(cfg, n)
        self.mask = np.zeros(self.L.total_bytes, bool)
        L, W = self.L, cfg.window
        self.sizes = dict(codes=128 * 128 * cfg.code_bits // 8, sigma=512, lambda_=512,
                          comp_id=4 * L.comp_id_stride, comp_line=512 * cfg.n_comp)

    def allow(self, off, nbytes):
        self.mask[off:off + nbytes] = True

    def header(self):
        self.allow(0, 48)

    def counts(self, states):
        for s in states:
            self.allow(self.L.counts + 4 * s, 4)

    def boundary(self, states):
        for s in states:
            for plane, b in self.sizes.items():
                self.allow(getattr(self.L, plane) + s * b, b)

    def record(self, states, slots):
        W, L = self.cfg.window, self.L
        for s, m in zip(states, slots):
            self.allow(L.rec_k + (s * W + m) * 512, 512)
            self.allow(L.rec_u + (s * W + m) * 512, 512)
            if self.cfg.decay_per_key:
                self.allow(L.rec_alpha + (s * W + m) * 512, 512)
            else:
                self.allow(L.rec_alpha + (s * L.alpha_stride + m) * 4, 4)

    def full_list(self):
        self.allow(self.L.full_list, 4 * self.n)


def _check_call(st, inputs, outputs, regions):
    changed = (st.inner != st.snap).cpu().numpy()
    stray = np.flatnonzero(changed & ~regions.mask)
    assert stray.size == 0, f"{stray.size} bytes written outside the call's work, first at {stray[:8]}"
    for g in [st] + inputs + outputs:
        assert g.guards_ok()
    for g in inputs:
        assert torch.equal(g.inner, g.snap)
    st.snap = st.inner.clone()
    for g in outputs:
        g.snap = g.inner.clone()


@pytest.mark.parametrize("n", [1, 3, 33, 157])
@pytest.mark.parametrize("kda,bits", [(False, 8), (True, 4)])
def test_calls_write_only_their_own_bytes(n, kda, bits):
    W, C = 4, 3
    cfg = lq.config(window=W, n_comp=C, kda=kda, code_bits=bits)
    wl = wlm.custom(900 + n + 7 * kda, n, 0, kda=kda, n_warm=12, plant=True)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, 16)
    st = Guarded(lq.state_bytes(cfg, n), np.full(lq.state_bytes(cfg, n), PAT, np.uint8))
    s0 = Guarded(S0.nbytes, S0)
    o = Guarded(n * 512)
    counts = np.zeros(n, int)
    allst = range(n)

    def token(t):
        ins = [Guarded(x.nbytes, x) for x in tk.token(t)]
        return ins, [g.f32() for g in ins]

    # whole-buffer init: header fields, counts, every boundary
    r = Regions(cfg, n)
    r.header(); r.counts(allst); r.boundary(allst)
    lq.state_init(cfg, st.inner, n, s0.f32())
    _check_call(st, [s0], [], r)
    # stated phases: three appends, then the fused last token (fold)
    for t in range(W):
        ins, x = token(t)
        r = Regions(cfg, n)
        r.counts(allst); r.record(allst, counts)
        if t == W - 1:
            r.boundary(allst)
        lq.decode_step(cfg, st.inner, n, *x, o.f32(), phase=t)
        _check_call(st, ins, [o], r)
        counts = (counts + 1) % W
    # mixed phases: one step, a range re-admitted, three more steps (the last folds the rest)
    first, cnt = n // 3, max(1, n // 3)
    for t in range(W, 2 * W):
        if t == W + 1:
            r = Regions(cfg, n)
            rng = range(first, first + cnt)
            r.counts(rng); r.boundary(rng)
            lq.state_init_range(cfg, st.inner, n, first, cnt, s0.f32()[first * 16384:(first + cnt) * 16384])
            _check_call(st, [s0], [], r)
            counts[first:first + cnt] = 0
        ins, x = token(t)
        r = Regions(cfg, n)
        r.counts(allst); r.record(allst, counts); r.full_list()
        r.boundary([s for s in allst if counts[s] == W - 1])
        lq.decode_step(cfg, st.inner, n, *x, o.f32())
        _check_call(st, ins, [o], r)
        counts = (counts + 1) % W
    # lq_fold with any counts
    r = Regions(cfg, n)
    r.counts(allst); r.boundary(allst)
    lq.fold(cfg, st.inner, n)
    _check_call(st, [], [], r)
    counts[:] = 0
    # two records per token: the second token fills every window (list fold)
    for t in range(2 * W, 2 * W + 4, 2):
        ins, x = token(t)
        ins2, x2 = token(t + 1)
        r = Regions(cfg, n)
        r.counts(allst); r.full_list()
        r.record(allst, counts); r.record(allst, counts + 1)
        r.boundary([s for s in allst if counts[s] + 2 == W])
        if kda:
            q, kh, _, w, _ = x
            _, k, v, a, _ = x2
            lq.decode_step_rwkv7(cfg, st.inner, n, q, w, kh, a, k, v, o.f32())
        else:
            q, k1, v1, a, b1 = x
            _, k2, v2, _, b2 = x2
            lq.decode_step2(cfg, st.inner, n, q, k1, v1, b1, k2, v2, b2, a, o.f32())
        _check_call(st, ins + ins2, [o], r)
        counts = (counts + 2) % W
    # export with records held: the state buffer is not written at all
    ins, x = token(2 * W + 4)
    r = Regions(cfg, n)
    r.counts(allst); r.record(allst, counts)
    lq.decode_step(cfg, st.inner, n, *x, o.f32(), phase=0)
    _check_call(st, ins, [o], r)
    out = Guarded(n * 16384 * 4)
    lq.export_state(cfg, st.inner, n, out.f32())
    _check_call(st, [], [out], Regions(cfg, n))
    assert lq.get_status(st.inner) == (lq.OK, -1)
