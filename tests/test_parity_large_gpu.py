"""A state buffer far past 4 GiB (262,144 head-states at W = 16, C = 4: 8.8 GiB), so every
byte offset the kernels form for the later head-states lies beyond 2^32 and must be
64-bit. The head-states are B distinct ones repeated R times: head-state s takes the
initial state and the tokens of head-state s mod B. Head-states are independent, so
every repeat must end bit-identical to the first block in o after every token and in
every plane of the buffer after every fold, a property that holds at any size; an
offset that wrapped would make a repeat read or write another head-state's bytes. The
first block's sampled head-states are held to the oracle as in the other parity tests,
so through the property the last head-states are too. A window of stated phases
(ending in the fused step) is followed by a mixed-phase window (the work list and the
list fold over all 262,144 head-states) and one more token.
"""
import numpy as np
import pytest
import torch

from oracle import FoldDiag, OracleState
from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import DEV, Tally, compare_boundary, to_dev, unpack_codes
from tests._helpers import rel_l2

pytestmark = pytest.mark.gpu

B, R = 1024, 256
W, C = 16, 4
SAMPLE = [0, 1, 517, B - 1]


def _plane_bytes(cfg, L):
    """(offset, bytes per head-state) of every per-head-state plane except the work list."""
    D = cfg.d_k
    return [(L.counts, 4), (L.codes, D * D * cfg.code_bits // 8), (L.sigma, 4 * D), (L.lambda_, 4 * D),
            (L.comp_id, 4 * L.comp_id_stride), (L.comp_line, 4 * cfg.n_comp * D), (L.rec_k, 4 * cfg.window * D),
            (L.rec_u, 4 * cfg.window * D), (L.rec_alpha, 4 * L.alpha_stride)]


def _assert_repeats_equal(state, planes, n, what):
    for off, per in planes:
        x = state[off:off + n * per].view(R, B * per)
        for r0 in range(1, R, 64):
            r1 = min(R, r0 + 64)
            assert torch.equal(x[r0:r1], x[:1].expand(r1 - r0, -1)), (what, off, r0)


def test_state_past_4gib_repeats_bit_identical_and_matches_oracle():
    n = B * R
    cfg = lq.config(window=W, n_comp=C)
    L = lq.layout(cfg, n)
    assert L.total_bytes > 2 * 2**32 and L.rec_alpha + n * 4 * L.alpha_stride > 2**33
    wl = wlm.custom(540, B, 0, n_warm=40, plant=True)
    S0, _ = wlm.initial_state(wl)
    n_tok = 2 * W + 1
    tk = wlm.tokens(wl, 0, n_tok)
    sub = tk.select_states(SAMPLE)

    state = torch.zeros(L.total_bytes, dtype=torch.uint8, device=DEV)  # padding never written reads 0 everywhere
    lq.state_init(cfg, state, n, None)
    S0d = to_dev(S0)
    for r in range(R):
        lq.state_init_range(cfg, state, n, r * B, B, S0d)
    del S0d
    planes = _plane_bytes(cfg, L)
    views = lq.state_views(cfg, state, n)
    sidx = torch.as_tensor(SAMPLE, device=DEV)
    last = torch.as_tensor([n - B + i for i in SAMPLE], device=DEV)

    ref = OracleState(len(SAMPLE), W=W, C=C)
    d0 = [FoldDiag(128, 128) for _ in SAMPLE]
    ref.init(S0[SAMPLE], diags=d0)
    tally = Tally()

    def boundary(idx):
        return dict(codes=unpack_codes(views["codes"][idx].cpu().numpy()), sigma=views["sigma"][idx].cpu().numpy(),
                    lam=views["lambda"][idx].cpu().numpy(), comp_id=views["comp_id"][idx].cpu().numpy(),
                    comp_line=views["comp_line"][idx].cpu().numpy(), count=views["counts"][idx].cpu().numpy())

    torch.cuda.synchronize()
    _assert_repeats_equal(state, planes, n, "init")
    compare_boundary(boundary(last), ref, range(len(SAMPLE)), d0, tally, "init")

    o = torch.empty((n, 128), dtype=torch.float32, device=DEV)
    for t in range(n_tok):
        q, k, v, a, b = (to_dev(x[t]).repeat((R,) + (1,) * (x.ndim - 2)) for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta))
        phase = t % W if (t < W or t == 2 * W) else lq.PHASE_ANY
        lq.decode_step(cfg, state, n, q, k, v, a, b, o, phase=phase)
        del q, k, v, a, b
        ov = o.view(R, B, 128)
        assert torch.equal(ov.view(torch.int32), ov[:1].view(torch.int32).expand(R, -1, -1)), f"o at token {t}"
        o_ref = ref.run(*(x[t:t + 1] for x in (sub.q, sub.k, sub.v, sub.alpha, sub.beta)), fold_when_full=False)[0]
        err = rel_l2(o.index_select(0, sidx).cpu().numpy(), o_ref)
        assert err.max() <= 1e-4, (t, err.max())
        slot = t % W
        assert np.array_equal(views["rec_u"].index_select(0, last)[:, slot].cpu().numpy(), ref.rec_u[:, slot]), t
        if (t + 1) % W == 0:
            dg = [FoldDiag(128, 128) for _ in SAMPLE]
            ref.fold(diags=dg)
            torch.cuda.synchronize()
            _assert_repeats_equal(state, planes, n, f"fold at token {t}")
            compare_boundary(boundary(last), ref, range(len(SAMPLE)), dg, tally, f"fold at token {t}")
    torch.cuda.synchronize()
    _assert_repeats_equal(state, planes, n, "end")
    status, bad = lq.get_status(state)
    assert status == lq.OK, (lq.STATUS_NAMES.get(status), bad)
    tally.check()
