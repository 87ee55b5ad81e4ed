"""4-bit codes (LeapQuant §4 evaluates 8-, 6- and 4-bit states; this build runs 8
and 4 on the GPU) against the oracle at the same code width: the same bit-exact
bar as 8-bit codes (codes and compensators exact except at rounding ties,
outputs within 1e-4 relative L2)."""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import DEV, GpuState, Tally, run_and_compare, to_dev, unpack_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_4bit_tiny(phase_mode):
    run_and_compare(wlm.WORKLOADS[1], 64, phase_mode=phase_mode, code_bits=4)


@pytest.mark.parametrize("n", [1, 33, 157])
def test_4bit_ragged_warm_planted(n):
    wl = wlm.custom(600 + n, n, 0, n_warm=96, plant=True)
    run_and_compare(wl, 40, code_bits=4)


def test_4bit_kda():
    wl = wlm.custom(610, 9, 0, kda=True, vdist="t3", n_warm=64)
    run_and_compare(wl, 36, code_bits=4)


@pytest.mark.parametrize("W,C,smooth", [(7, 3, True), (16, 0, False), (32, 8, True)])
def test_4bit_window_and_compensator_variants(W, C, smooth):
    wl = wlm.custom(620 + W + C, 11, 0, n_warm=48, plant=True)
    run_and_compare(wl, 2 * W + 3, W=W, C=C, smooth=smooth, code_bits=4)


def test_4bit_batch512_full_size_sampled():
    wl = wlm.WORKLOADS[4]
    tally = run_and_compare(wl, 48, sample=[0, 5, 4097, 9999, wl.n_states - 1], chunk=48, code_bits=4)
    assert tally.entries > 0


def test_4bit_codes_stay_in_range_and_fold_separately():
    wl = wlm.custom(630, 5, 0, n_warm=32, plant=True)
    S0, _ = wlm.initial_state(wl)
    g = GpuState(5, code_bits=4)
    g.init(S0)
    tk = wlm.tokens(wl, 0, 5)
    for t in range(5):
        g.append(*(to_dev(x) for x in tk.token(t)))
    g.fold()
    codes = unpack_codes(g.views["codes"].cpu().numpy())
    assert codes.min() >= -7 and codes.max() <= 7
    raw = g.views["codes"].cpu().numpy()
    assert ((raw & 0x0F) >= 1).all() and ((raw >> 4) >= 1).all()  # stored c + 8 is never 0
    assert g.status()[0] == lq.OK
