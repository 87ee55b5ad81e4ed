"""RWKV7 tokens (lq_decode_step_rwkv7) against the oracle.

LeapQuant App. A splits an RWKV7 token, whose erase direction differs from its
write key, into an erase and a pure-write sub-step: records (a . kh, -(S kh), w)
and (k, v, 1). The oracle's form is pinned against RWKV7's update in
test_oracle_rwkv.py; the GPU builds both records in one kernel. Same bar as
the other tokens: records and codes exact (codes except at rounding ties),
outputs within 1e-4 relative L2.
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


class RwkvTokens:
    """RWKV7 token t from generator tokens 2t (decay w, erase direction kh) and 2t+1
    (receptance r, rate a, write key k, value v); kh normalized in fp32."""

    def __init__(self, wl, n, states=None):
        tk = wlm.tokens(wl, 0, 2 * n, states=states)
        kh = tk.k[0::2]
        self.kh = (kh / np.linalg.norm(kh, axis=-1, keepdims=True)).astype(np.float32)
        self.w, self.a = tk.alpha[0::2], tk.alpha[1::2]
        self.r, self.k, self.v = tk.q[1::2], tk.k[1::2], tk.v[1::2]

    def args(self, t, idx=slice(None)):
        return [x[t][idx] for x in (self.r, self.w, self.kh, self.a, self.k, self.v)]


def run_rwkv(wl, n_tokens, W=16, C=4, phase_mode="stated", code_bits=8, comp_fit=0, comp_block=0, sample=None):
    assert wl.kda
    N = wl.n_states
    sample = list(range(N)) if sample is None else list(sample)
    S0, _ = wlm.initial_state(wl)
    gpu = GpuState(N, W=W, C=C, kda=True, code_bits=code_bits, comp_fit=comp_fit, comp_block=comp_block)
    gpu.init(S0)
    ref = OracleState(len(sample), W=W, C=C, decay_per_key=True, code_bits=code_bits, comp_fit=comp_fit,
                      comp_block=comp_block)
    ref.init(None if S0 is None else S0[sample])
    sidx = torch.as_tensor(sample, device=DEV)
    tally = Tally()
    tt = RwkvTokens(wl, n_tokens)
    for t in range(n_tokens):
        n0 = (2 * t) % W
        phase = n0 if phase_mode == "stated" else lq.PHASE_ANY
        lq.decode_step_rwkv7(gpu.cfg, gpu.state, N, *(to_dev(x) for x in tt.args(t)), gpu.o, phase=phase)
        o_ref = ref.append_rwkv(*tt.args(t, sample))
        err = rel_l2(gpu.o.index_select(0, sidx).cpu().numpy(), o_ref)
        tally.worst_o = max(tally.worst_o, float(err.max()))
        assert err.max() <= 1e-4, (t, err.max())
        ru = gpu.views["rec_u"].index_select(0, sidx).cpu().numpy()
        rk = gpu.views["rec_k"].index_select(0, sidx).cpu().numpy()
        ra = gpu.views["rec_alpha"].index_select(0, sidx).cpu().numpy().reshape(len(sample), W, 128)
        for slot in (n0, n0 + 1):
            assert np.array_equal(ru[:, slot], ref.rec_u[:, slot]), (t, slot)
            assert np.array_equal(rk[:, slot], ref.rec_k[:, slot]), (t, slot)
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
def test_rwkv_tiny(phase_mode):
    run_rwkv(wlm.custom(900, 2, 0, kda=True, n_warm=32), 24, phase_mode=phase_mode)


@pytest.mark.parametrize("n", [1, 33])
def test_rwkv_ragged_warm_planted(n):
    run_rwkv(wlm.custom(910 + n, n, 0, kda=True, vdist="t3", n_warm=96, plant=True), 20)


@pytest.mark.parametrize("code_bits,comp_fit,comp_block", [(6, 0, 0), (4, 0, 0), (8, 2, 0), (8, 2, 1)])
def test_rwkv_code_width_and_compensator_forms(code_bits, comp_fit, comp_block):
    wl = wlm.custom(920 + code_bits + comp_fit + comp_block, 9, 0, kda=True, n_warm=48, plant=True)
    run_rwkv(wl, 14, W=6, C=2, code_bits=code_bits, comp_fit=comp_fit, comp_block=comp_block)


def test_rwkv_window_of_two_and_thirty_two():
    wl = wlm.custom(930, 5, 0, kda=True, n_warm=32, plant=True)
    run_rwkv(wl, 5, W=2, C=1)
    run_rwkv(wl, 20, W=32, C=8)


def test_rwkv_kda_workload_full_size_sampled():
    wl = wlm.WORKLOADS[5]
    tally = run_rwkv(wl, 10, sample=[0, 777, 30000, wl.n_states - 1])
    assert tally.entries > 0


def test_rwkv_needs_per_key_decay():
    g = GpuState(2)  # scalar decay
    g.init(None)
    x = torch.zeros(2, 128, device=DEV)
    with pytest.raises(lq.LQError) as e:
        lq.decode_step_rwkv7(g.cfg, g.state, 2, x, x, x, x, x, x, torch.empty(2, 128, device=DEV))
    assert e.value.code == lq.ERR_UNSUPPORTED
