"""Head-states at different window phases: requests admitted at different tokens.

LeapQuant's windows belong to each head-state (§3.2 Per-window quantization:
the boundary stays fixed for W tokens of that state, then one fold rounds it),
so nothing ties the windows of different requests together. Here
lq_state_init_range re-admits groups of head-states at different tokens, and
lq_decode_step with LQ_PHASE_ANY then appends every head-state and folds the
ones whose own window filled (the append lists them, a second kernel folds the
list). The bar is the in-phase one: codes and compensators exact except at
rounding ties, outputs within 1e-4 relative L2, records exact.
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


def _groups(n, g, seed):
    """Cut 0..n into g contiguous groups of ragged sizes (every group non-empty when n >= g)."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, n), size=min(g, n) - 1, replace=False)) if n > 1 else np.array([], int)
    return [0] + [int(c) for c in cuts] + [n]


def _header_words(state):
    """(full_n, fold_done) of the state buffer's header: the work list is empty between calls."""
    h = state[:48].cpu().numpy()
    return int(h[40:44].view(np.int32)[0]), int(h[44:48].view(np.int32)[0])


def run_staggered(wl, n_tokens, bounds, W=16, C=4, code_bits=8, comp_fit=0, sample=None, admit_every=1):
    """Decode n_tokens for all head-states; group g >= 1 (states bounds[g]..bounds[g+1]-1)
    is re-admitted from a second initial state before token g * admit_every. The oracle
    follows the sampled states (all by default)."""
    N = wl.n_states
    sample = list(range(N)) if sample is None else sorted(sample)
    pos = {s: i for i, s in enumerate(sample)}
    S0, _ = wlm.initial_state(wl)
    wl1 = wlm.custom(wl.wid + 5000, N, 0, kda=wl.kda, n_warm=48, plant=True)
    S1, _ = wlm.initial_state(wl1)
    gpu = GpuState(N, W=W, C=C, kda=wl.kda, code_bits=code_bits, comp_fit=comp_fit)
    gpu.init(S0)
    ref = OracleState(len(sample), W=W, C=C, decay_per_key=wl.kda, code_bits=code_bits, comp_fit=comp_fit)
    ref.init(None if S0 is None else S0[sample])
    sidx = torch.as_tensor(sample, device=DEV)
    tally = Tally()
    admitted = 0
    folds = np.zeros(n_tokens, np.int64)
    tk = wlm.tokens(wl, 0, n_tokens)
    sub = tk.select_states(sample)
    for t in range(n_tokens):
        for g in range(1, len(bounds) - 1):
            if t != g * admit_every:
                continue
            a, b = bounds[g], bounds[g + 1]
            lq.state_init_range(gpu.cfg, gpu.state, N, a, b - a, to_dev(S1[a:b]))
            mine = [s for s in sample if a <= s < b]
            if mine:
                d = [FoldDiag(128, 128) for _ in mine]
                first = pos[mine[0]]
                ref.init_range(first, len(mine), S1[mine], diags=d)
                compare_boundary(gpu.boundary(mine), ref, range(first, first + len(mine)), d, tally,
                                 f"admission of group {g} at token {t}")
            admitted += 1
        q, k, v, al, be = (to_dev(x) for x in tk.token(t))
        gpu.step(q, k, v, al, be, phase=lq.PHASE_ANY)
        o_ref = ref.run(*(x[t:t + 1] for x in (sub.q, sub.k, sub.v, sub.alpha, sub.beta)), fold_when_full=False)[0]
        err = rel_l2(gpu.o.index_select(0, sidx).cpu().numpy(), o_ref)
        tally.worst_o = max(tally.worst_o, float(err.max()))
        assert err.max() <= 1e-4, (t, err.max())
        full = [i for i in range(len(sample)) if ref.count[i] == W]
        if full:
            dg = [FoldDiag(128, 128) for _ in full]
            ref.fold(states=full, diags=dg)
            compare_boundary(gpu.boundary([sample[i] for i in full]), ref, full, dg, tally, f"fold at token {t}")
        counts = gpu.views["counts"].cpu().numpy()
        assert np.array_equal(counts[sample], ref.count), t
        assert counts.max() < W  # every window that filled was folded in the same call
        folds[t] = len(full)
    st, bad = gpu.status()
    assert st == lq.OK, (lq.STATUS_NAMES.get(st), bad)
    assert _header_words(gpu.state) == (0, 0)
    assert np.array_equal(gpu.export(sample), ref.export())
    tally.check()
    return tally, folds


def test_staggered_gdn_ragged_groups():
    """45 head-states in 16 ragged groups, one admitted per token: from token 16 on
    every window phase is present and some head-states fold at nearly every token."""
    wl = wlm.custom(700, 45, 0, n_warm=64, plant=True)
    bounds = _groups(45, 16, 1)
    _, folds = run_staggered(wl, 52, bounds)
    assert (folds[16:] > 0).mean() > 0.8


def test_staggered_kda_short_window():
    wl = wlm.custom(710, 19, 0, kda=True, vdist="t3", n_warm=48)
    _, folds = run_staggered(wl, 30, _groups(19, 7, 2), W=7, C=3)
    assert folds.sum() > 0


@pytest.mark.parametrize("code_bits,comp_fit", [(4, 0), (8, 3)])
def test_staggered_code_width_and_fitted_factors(code_bits, comp_fit):
    wl = wlm.custom(720 + code_bits + comp_fit, 13, 0, n_warm=40, plant=True)
    run_staggered(wl, 26, _groups(13, 8, 3), W=8, C=2, code_bits=code_bits, comp_fit=comp_fit)


def test_single_state_and_more_groups_than_tokens_in_a_window():
    """n = 1 (the list fold runs one CTA) and W = 1 (every token folds every head-state)."""
    wl = wlm.custom(730, 1, 0, n_warm=16, plant=True)
    run_staggered(wl, 5, [0, 1], W=4, C=1)
    wl = wlm.custom(731, 6, 0, n_warm=16, plant=True)
    _, folds = run_staggered(wl, 5, _groups(6, 3, 4), W=1, C=2)
    assert (folds == 6).all()


def test_staggered_batch512_full_size_sampled():
    """The benchmark's staggered workload: batch 512 (16,384 head-states) in 16 groups of
    1,024, group g admitted before token g; the oracle follows two states per group."""
    wl = wlm.WORKLOADS[4]
    N = wl.n_states
    bounds = [1024 * g for g in range(17)]
    sample = sorted({b + o for b in bounds[:-1] for o in (0, 1023)} | {N - 1})
    tally, folds = run_staggered(wl, 36, bounds, sample=sample)
    assert tally.entries > 0 and folds[16:].sum() > 0


def test_range_init_needs_a_matching_header_and_leaves_the_rest():
    n = 6
    gpu = GpuState(n)
    gpu.init(None)
    wl = wlm.custom(740, n, 0, n_warm=20, plant=True)
    tk = wlm.tokens(wl, 0, 3)
    for t in range(3):
        gpu.step(*(to_dev(x) for x in tk.token(t)), phase=t)
    before = gpu.state.clone()
    S1, _ = wlm.initial_state(wl)
    lq.state_init_range(gpu.cfg, gpu.state, n, 2, 3, to_dev(S1[2:5]))
    assert gpu.views["counts"].tolist() == [3, 3, 0, 0, 0, 3]
    assert gpu.status()[0] == lq.OK
    ref = OracleState(3)
    d = [FoldDiag(128, 128) for _ in range(3)]
    ref.init(S1[2:5], diags=d)
    compare_boundary(gpu.boundary([2, 3, 4]), ref, range(3), d, None, "range init")
    bv = lq.state_views(gpu.cfg, before, n)
    for name in ("codes", "sigma", "lambda", "comp_id", "comp_line", "rec_k", "rec_u", "rec_alpha"):
        for st in (0, 1, 5):
            assert torch.equal(gpu.views[name][st], bv[name][st]), (name, st)
    # an empty range does nothing; a buffer set up for another n_states is refused on the device
    lq.state_init_range(gpu.cfg, gpu.state, n, 6, 0, None)
    snap = gpu.state.clone()
    lq.state_init_range(gpu.cfg, gpu.state, n - 1, 0, 2, None)
    status, bad = gpu.status()
    assert status == lq.ERR_STATE and bad in (0, 1)
    lay = lq.layout(gpu.cfg, n)
    assert torch.equal(gpu.state[lay.counts:], snap[lay.counts:])


def test_any_phase_with_a_full_window_leaves_it_and_the_list_empty():
    """A head-state filled by lq_append is not appended to by a mixed-phase step (status
    LQ_ERR_WINDOW_FULL), is not folded, and the work list ends empty."""
    cfg = lq.config(window=3)
    n = 5
    st = lq.alloc_state(cfg, n, DEV)
    lq.state_init(cfg, st, n, None)
    wl = wlm.custom(750, n, 0)
    tk = wlm.tokens(wl, 0, 4)
    o = torch.empty(n, 128, device=DEV)
    for t in range(3):
        lq.append(cfg, st, n, *(to_dev(x) for x in tk.token(t)), o)
    lq.state_init_range(cfg, st, n, 1, 2, None)  # states 1, 2 restart; 0, 3, 4 stay full
    lay = lq.layout(cfg, n)
    full_before = [st[lay.rec_k:lay.rec_u].clone()]
    lq.decode_step(cfg, st, n, *(to_dev(x) for x in tk.token(3)), o)
    status, bad = lq.get_status(st)
    assert status == lq.ERR_WINDOW_FULL and bad in (0, 3, 4)
    assert lq.state_views(cfg, st, n)["counts"].tolist() == [3, 1, 1, 3, 3]
    assert _header_words(st) == (0, 0)
    rk = lq.state_views(cfg, st, n)["rec_k"]
    rk0 = full_before[0].view(torch.float32).view(n, 3, 128)
    for s in (0, 3, 4):
        assert torch.equal(rk[s], rk0[s])
