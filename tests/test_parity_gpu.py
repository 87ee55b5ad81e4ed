"""GPU vs oracle parity through the C ABI (free-running, element by element).

Outputs o within 1e-4 relative L2 per (head-state, token); int8 codes and
compensator ids bit-exact except codes within 1e-6 relative of a rounding tie
(fewer than 1e-5 of entries, at most one code apart); sigma, lambda, compensator
lines, record u and the exported state bit-exact.
"""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_tiny_gdn_workload_full(phase_mode):
    from tests._gpu import run_and_compare

    wl = wlm.WORKLOADS[1]
    run_and_compare(wl, wl.n_tokens, phase_mode=phase_mode)


@pytest.mark.parametrize("n", [1, 3, 33, 157, 305])
def test_ragged_batches_warm_planted(n):
    from tests._gpu import run_and_compare

    wl = wlm.custom(200 + n, n, 0, n_warm=48, plant=True)
    run_and_compare(wl, 2 * 16 + 5)


def test_kda_t3_small():
    from tests._gpu import run_and_compare

    wl = wlm.WORKLOADS[5]
    small = wlm.Workload(wl.wid, wl.name, 6, 40, True, "t3", 512, False, 1, 1, 6)
    run_and_compare(small, small.n_tokens)


@pytest.mark.parametrize("W,C,smooth", [(1, 0, False), (7, 3, True), (32, 8, True), (16, 4, False), (5, 0, True)])
def test_window_and_compensator_variants(W, C, smooth):
    from tests._gpu import run_and_compare

    wl = wlm.custom(300 + W * 10 + C, 9, 0, n_warm=32, plant=True)
    run_and_compare(wl, 2 * W + 3, W=W, C=C, smooth=smooth)


def test_kda_variants():
    from tests._gpu import run_and_compare

    wl = wlm.custom(390, 5, 0, kda=True, vdist="t3", n_warm=40)
    run_and_compare(wl, 2 * 7 + 2, W=7, C=5)


def test_separate_append_and_fold_match_fused_step():
    from tests._gpu import run_and_compare

    wl = wlm.custom(400, 11, 0, n_warm=40, plant=True)
    run_and_compare(wl, 2 * 16 + 4, use_append_fold=True)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_exact_ties_round_to_even(bits):
    """The init-fold's rounding at exact half-integers (reading R8: half to even), the
    same typed-out codes the oracle is pinned to; then a fold with no records keeps them."""
    from tests._gpu import GpuState, to_dev
    from tests._helpers import tie_rows

    qm = 2 ** (bits - 1) - 1
    S0, want = tie_rows(qm)
    g = GpuState(1, C=0, smooth=False, code_bits=bits)
    g.init(S0)
    b = g.boundary()
    assert np.array_equal(b["codes"], want)
    assert np.array_equal(b["sigma"][0, :3], (np.float32(qm) * np.float32([0.5, 1.0, 2.0])) / np.float32(qm))
    g.fold()
    assert np.array_equal(g.boundary()["codes"], want)
    assert g.status()[0] == lq.OK


@pytest.mark.parametrize("case", range(3))
def test_selection_exact_score_ties(case):
    """The init-fold and a later fold on states whose compensator selection meets exact
    score ties: the hand-worked ids of the oracle's pin, and the whole boundary bit-exact."""
    from oracle import FoldDiag, OracleState
    from tests._gpu import GpuState, compare_boundary
    from tests._helpers import selection_ties

    S0, want = selection_ties()[case]
    g = GpuState(1)
    g.init(S0)
    ref = OracleState(1, W=16, C=4)
    dg = [FoldDiag(128, 128)]
    ref.init(S0, diags=dg)
    b = g.boundary()
    assert b["comp_id"][0, :4].tolist() == want
    compare_boundary(b, ref, [0], dg, what="init")
    g.fold()
    dg = [FoldDiag(128, 128)]
    ref.fold(diags=dg)
    compare_boundary(g.boundary(), ref, [0], dg, what="fold")
    assert g.status()[0] == lq.OK
