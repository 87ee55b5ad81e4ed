"""Two-record tokens (lq_decode_step2) against the oracle.

LeapQuant App. A: a token whose update takes two rank-one sub-steps leaves two
records; in the DeltaProduct form the second record has decay 1. The oracle
runs the two sub-steps as two appends (pinned against the product form in
test_oracle_two_record.py); the GPU runs them in one kernel with one read of
the boundary. Same bar as one-record tokens: records and codes exact (codes
except at rounding ties), outputs within 1e-4 relative L2.
"""
import numpy as np
import pytest
import torch

from oracle import FoldDiag, OracleState
from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import DEV, GpuState, Tally, compare_boundary, to_dev
from tests._helpers import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


class TwoTokens:
    """Token t of a two-record stream: sub-step 1 from generator token 2t (k1, v1,
    beta1, alpha), sub-step 2 and the query from generator token 2t+1."""

    def __init__(self, wl, t0, n, states=None):
        tk = wlm.tokens(wl, 2 * t0, 2 * n, states=states)
        self.q, self.k2, self.v2, self.b2 = tk.q[1::2], tk.k[1::2], tk.v[1::2], tk.beta[1::2]
        self.k1, self.v1, self.b1, self.a = tk.k[0::2], tk.v[0::2], tk.beta[0::2], tk.alpha[0::2]

    def dev(self, t):
        return [to_dev(x[t]) for x in (self.q, self.k1, self.v1, self.b1, self.k2, self.v2, self.b2, self.a)]

    def sub(self, idx):
        out = object.__new__(TwoTokens)
        for f in ("q", "k1", "v1", "b1", "k2", "v2", "b2", "a"):
            setattr(out, f, getattr(self, f)[:, idx])
        return out


def run_two(wl, n_tokens, W=16, C=4, phase_mode="stated", code_bits=8, comp_fit=0, sample=None):
    N = wl.n_states
    sample = list(range(N)) if sample is None else list(sample)
    S0, _ = wlm.initial_state(wl)
    gpu = GpuState(N, W=W, C=C, kda=wl.kda, code_bits=code_bits, comp_fit=comp_fit)
    gpu.init(S0)
    ref = OracleState(len(sample), W=W, C=C, decay_per_key=wl.kda, code_bits=code_bits, comp_fit=comp_fit)
    ref.init(None if S0 is None else S0[sample])
    sidx = torch.as_tensor(sample, device=DEV)
    tally = Tally()
    tt = TwoTokens(wl, 0, n_tokens)
    sub = tt.sub(sample)
    ones = np.ones_like(sub.a[0])
    for t in range(n_tokens):
        n0 = (2 * t) % W
        phase = n0 if phase_mode == "stated" else lq.PHASE_ANY
        q, k1, v1, b1, k2, v2, b2, a = tt.dev(t)
        lq.decode_step2(gpu.cfg, gpu.state, N, q, k1, v1, b1, k2, v2, b2, a, gpu.o, phase=phase)
        ref.run(sub.q[t][None], sub.k1[t][None], sub.v1[t][None], sub.a[t][None], sub.b1[t][None],
                fold_when_full=False)
        o_ref = ref.run(sub.q[t][None], sub.k2[t][None], sub.v2[t][None], ones[None], sub.b2[t][None],
                        fold_when_full=False)[0]
        err = rel_l2(gpu.o.index_select(0, sidx).cpu().numpy(), o_ref)
        tally.worst_o = max(tally.worst_o, float(err.max()))
        assert err.max() <= 1e-4, (t, err.max())
        ru = gpu.views["rec_u"].index_select(0, sidx).cpu().numpy()
        ra = gpu.views["rec_alpha"].index_select(0, sidx).cpu().numpy()
        ra = ra.reshape(len(sample), W, 128) if wl.kda else ra[:, :W, None]
        for slot in (n0, n0 + 1):
            assert np.array_equal(ru[:, slot], ref.rec_u[:, slot]), (t, slot)
            assert np.array_equal(ra[:, slot], ref.rec_alpha[:, slot]), (t, slot)
        if n0 + 2 == W:
            dg = [FoldDiag(128, 128) for _ in sample]
            ref.fold(diags=dg)
            compare_boundary(gpu.boundary(sample), ref, range(len(sample)), dg, tally, f"fold at token {t}")
        assert np.array_equal(gpu.views["counts"].index_select(0, sidx).cpu().numpy(), ref.count), t
    st, bad = gpu.status()
    assert st == lq.OK, (lq.STATUS_NAMES.get(st), bad)
    assert np.array_equal(gpu.export(sample), ref.export())
    tally.check()
    return tally


@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_two_record_tiny(phase_mode):
    run_two(wlm.WORKLOADS[1], 24, phase_mode=phase_mode)


@pytest.mark.parametrize("n", [1, 33, 157])
def test_two_record_ragged_warm_planted(n):
    wl = wlm.custom(800 + n, n, 0, n_warm=96, plant=True)
    run_two(wl, 20)


def test_two_record_kda():
    wl = wlm.custom(810, 9, 0, kda=True, vdist="t3", n_warm=64)
    run_two(wl, 18, W=8, C=3)


@pytest.mark.parametrize("code_bits,comp_fit", [(4, 0), (8, 3)])
def test_two_record_code_width_and_fitted_factors(code_bits, comp_fit):
    wl = wlm.custom(820 + code_bits + comp_fit, 11, 0, n_warm=48, plant=True)
    run_two(wl, 14, W=6, C=2, code_bits=code_bits, comp_fit=comp_fit)


def test_two_record_window_of_two_and_thirty_two():
    """W = 2: every token fills and folds the window; W = 32: the key prefetch covers
    16 records and the rest are read from global memory."""
    wl = wlm.custom(830, 5, 0, n_warm=32, plant=True)
    run_two(wl, 5, W=2, C=1)
    run_two(wl, 20, W=32, C=8)


def test_two_record_batch512_full_size_sampled():
    wl = wlm.WORKLOADS[4]
    tally = run_two(wl, 12, sample=[0, 5, 4097, 9999, wl.n_states - 1])
    assert tally.entries > 0


def test_two_record_tokens_mix_with_one_record_tokens():
    """A window may hold one- and two-record tokens in any order (LQ_PHASE_ANY)."""
    wl = wlm.custom(840, 7, 0, n_warm=24, plant=True)
    S0, _ = wlm.initial_state(wl)
    gpu = GpuState(7, W=8, C=2)
    gpu.init(S0)
    ref = OracleState(7, W=8, C=2)
    ref.init(S0)
    tt = TwoTokens(wl, 0, 10)
    ones = np.ones_like(tt.a[0])
    for t, kind in enumerate([2, 1, 2, 2, 1, 2, 1, 1, 2, 2]):
        q, k1, v1, b1, k2, v2, b2, a = tt.dev(t)
        if kind == 1:
            gpu.step(q, k1, v1, a, b1)
            o_ref = ref.run(tt.q[t][None], tt.k1[t][None], tt.v1[t][None], tt.a[t][None], tt.b1[t][None])[0]
        else:
            lq.decode_step2(gpu.cfg, gpu.state, 7, q, k1, v1, b1, k2, v2, b2, a, gpu.o)
            ref.run(tt.q[t][None], tt.k1[t][None], tt.v1[t][None], tt.a[t][None], tt.b1[t][None])
            o_ref = ref.run(tt.q[t][None], tt.k2[t][None], tt.v2[t][None], ones[None], tt.b2[t][None])[0]
        assert rel_l2(gpu.o.cpu().numpy(), o_ref).max() <= 1e-4, t
        assert gpu.views["counts"].tolist() == ref.count.tolist(), t
    assert gpu.status()[0] == lq.OK
    assert np.array_equal(gpu.export(), ref.export())


def test_two_record_token_without_room_sets_window_full():
    """W = 7: after three two-record tokens the window holds 6 records; a fourth does not
    fit, so the head-states are left unchanged and the status says so."""
    wl = wlm.custom(850, 4, 0)
    gpu = GpuState(4, W=7, C=1)
    gpu.init(None)
    tt = TwoTokens(wl, 0, 4)
    for t in range(3):
        lq.decode_step2(gpu.cfg, gpu.state, 4, *tt.dev(t), gpu.o, phase=2 * t)
    assert gpu.status()[0] == lq.OK
    lay = lq.layout(gpu.cfg, 4)
    before = gpu.state.clone()
    lq.decode_step2(gpu.cfg, gpu.state, 4, *tt.dev(3), gpu.o)
    status, bad = gpu.status()
    assert status == lq.ERR_WINDOW_FULL and 0 <= bad < 4
    assert torch.equal(gpu.state[lay.counts:], before[lay.counts:])
    with pytest.raises(lq.LQError) as e:
        lq.decode_step2(gpu.cfg, gpu.state, 4, *tt.dev(3), gpu.o, phase=6)
    assert e.value.code == lq.ERR_INVALID_ARG
