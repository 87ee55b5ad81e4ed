"""Parity at extreme magnitudes. The initial state and every v are multiplied by a
power of two on both sides (the same float32 inputs reach the GPU and the oracle).
At 2^-118 and 2^-124 the state, the record corrections and many products of the
fold and the append lie near or below the smallest normal float, so every kernel
path must keep subnormal values (no flush to zero) and round them as the oracle
does; the smoothing scales sit at their floor there. At 2^40 the squared line
lengths that rank the compensators reach about 2^107. Codes, ids, scales,
compensator lines and record corrections are held to the oracle bit for bit
(ties excepted, as everywhere), outputs within 1e-4 relative L2 in units of the
scale.
"""
import pytest

from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import run_and_compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("exp2", [-124, -118, 40])
@pytest.mark.parametrize("kda", [False, True])
def test_extreme_magnitudes(exp2, kda):
    wl = wlm.custom(570 + (exp2 % 97) + (7 if kda else 0), 33, 0, kda=kda, vdist="t3" if kda else "normal",
                    n_warm=40, plant=not kda)
    tally = run_and_compare(wl, 2 * wl.W + 3, scale=2.0 ** exp2)
    assert tally.entries > 0
