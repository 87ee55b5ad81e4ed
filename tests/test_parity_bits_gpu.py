"""6- and 4-bit codes (LeapQuant §4 evaluates 8-, 6- and 4-bit states) against the
oracle at the same code width: the same bit-exact bar as 8-bit codes (codes and
compensators exact except at rounding ties, outputs within 1e-4 relative L2)."""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import GpuState, run_and_compare, to_dev, unpack_codes

pytestmark = pytest.mark.gpu
BITS = [6, 4]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("phase_mode", ["stated", "any"])
def test_low_bit_tiny(bits, phase_mode):
    run_and_compare(wlm.WORKLOADS[1], 64, phase_mode=phase_mode, code_bits=bits)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("n", [1, 33, 157])
def test_low_bit_ragged_warm_planted(bits, n):
    wl = wlm.custom(600 + n, n, 0, n_warm=96, plant=True)
    run_and_compare(wl, 40, code_bits=bits)


@pytest.mark.parametrize("bits", BITS)
def test_low_bit_kda(bits):
    wl = wlm.custom(610, 9, 0, kda=True, vdist="t3", n_warm=64)
    run_and_compare(wl, 36, code_bits=bits)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("W,C,smooth", [(7, 3, True), (16, 0, False), (32, 8, True)])
def test_low_bit_window_and_compensator_variants(bits, W, C, smooth):
    wl = wlm.custom(620 + W + C, 11, 0, n_warm=48, plant=True)
    run_and_compare(wl, 2 * W + 3, W=W, C=C, smooth=smooth, code_bits=bits)


@pytest.mark.parametrize("bits", BITS)
def test_low_bit_batch512_full_size_sampled(bits):
    wl = wlm.WORKLOADS[4]
    tally = run_and_compare(wl, 48, sample=[0, 5, 4097, 9999, wl.n_states - 1], chunk=48, code_bits=bits)
    assert tally.entries > 0


def test_6bit_fitted_factors():
    wl = wlm.custom(625, 7, 0, n_warm=40, plant=True)
    run_and_compare(wl, 20, W=8, C=2, code_bits=6, comp_fit=3)


@pytest.mark.parametrize("bits", BITS)
def test_low_bit_codes_stay_in_range_and_fold_separately(bits):
    q = 2 ** (bits - 1) - 1
    wl = wlm.custom(630, 5, 0, n_warm=32, plant=True)
    S0, _ = wlm.initial_state(wl)
    g = GpuState(5, code_bits=bits)
    g.init(S0)
    tk = wlm.tokens(wl, 0, 5)
    for t in range(5):
        g.append(*(to_dev(x) for x in tk.token(t)))
    g.fold()
    raw = g.views["codes"].cpu().numpy()
    assert raw.shape == (5, 128, 128 * bits // 8)
    codes = unpack_codes(raw)
    assert codes.min() >= -q and codes.max() <= q
    assert (codes == -q).any() or (codes == q).any()  # every row's absmax maps to +-q
    lo = raw[..., :64]
    assert ((lo & 0x0F) >= (1 if bits == 4 else 0)).all()
    assert g.status()[0] == lq.OK
