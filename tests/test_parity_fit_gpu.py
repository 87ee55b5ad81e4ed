"""Fitted-factor compensators (comp_fit > 0: rank-one factors from power-iteration
sweeps; LeapQuant §3.3, App. B.3; research note 4) against the oracle: factors,
codes and scales bit-exact except at rounding ties, outputs within 1e-4. Both
fits: one factor at a time from the longest row, and the block fit that starts
each fold from the previous window's factors (research note 4, "Redesign")."""
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_fit_tiny(phase_mode):
    run_and_compare(wlm.WORKLOADS[1], 64, phase_mode=phase_mode, comp_fit=8)


@pytest.mark.parametrize("n", [3, 33])
def test_fit_warm_planted(n):
    wl = wlm.custom(700 + n, n, 0, n_warm=96, plant=True)
    run_and_compare(wl, 40, comp_fit=8)


def test_fit_kda():
    wl = wlm.custom(710, 5, 0, kda=True, vdist="t3", n_warm=64)
    run_and_compare(wl, 36, comp_fit=8)


@pytest.mark.parametrize("sweeps,C,bits", [(2, 4, 8), (8, 2, 4), (1, 8, 8)])
def test_fit_variants(sweeps, C, bits):
    wl = wlm.custom(720 + sweeps + C, 9, 0, n_warm=48, plant=True)
    run_and_compare(wl, 35, C=C, comp_fit=sweeps, code_bits=bits)


def test_fit_batch512_full_size_sampled():
    wl = wlm.WORKLOADS[4]
    run_and_compare(wl, 33, sample=[0, 1234, wl.n_states - 1], chunk=33, comp_fit=8)


@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_block_fit_tiny(phase_mode):
    run_and_compare(wlm.WORKLOADS[1], 64, phase_mode=phase_mode, comp_fit=2, comp_block=1)


@pytest.mark.parametrize("n", [1, 33])
def test_block_fit_warm_planted(n):
    wl = wlm.custom(740 + n, n, 0, n_warm=96, plant=True)
    run_and_compare(wl, 40, comp_fit=2, comp_block=1)


def test_block_fit_kda_and_lq_fold():
    wl = wlm.custom(750, 5, 0, kda=True, vdist="t3", n_warm=64)
    run_and_compare(wl, 36, comp_fit=1, comp_block=1)
    run_and_compare(wlm.custom(751, 6, 0, n_warm=32, plant=True), 34, comp_fit=3, comp_block=1, use_append_fold=True)


@pytest.mark.parametrize("sweeps,C,bits", [(1, 8, 8), (4, 3, 6), (2, 1, 4)])
def test_block_fit_variants(sweeps, C, bits):
    wl = wlm.custom(760 + sweeps + C, 9, 0, n_warm=48, plant=True)
    run_and_compare(wl, 35, C=C, comp_fit=sweeps, code_bits=bits, comp_block=1)


def test_block_fit_from_a_zero_state():
    """Zero initial states give zero factors; later folds fall back to the longest rows."""
    wl = wlm.custom(770, 4, 0)
    run_and_compare(wl, 40, comp_fit=2, comp_block=1)


def test_block_fit_batch512_full_size_sampled():
    wl = wlm.WORKLOADS[4]
    run_and_compare(wl, 33, sample=[0, 1234, wl.n_states - 1], chunk=33, comp_fit=2, comp_block=1)
