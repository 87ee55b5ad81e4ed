"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Every head-state of the workload runs on the GPU through lq_decode_step with the
stated window phase (the append-only kernel for 15 tokens, the fused
append+fold kernel for the 16th), free-running over the full token count. The
CPU oracle follows a sample of head-states (first, last and seeded others);
outputs are compared every token, record corrections every token, boundaries
after every fold and the exported state at the end.
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


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return sorted({0, n - 1, *map(int, rest)})


@pytest.mark.parametrize("wid", [2, 3, 4])
def test_gdn_workloads_full_size(wid):
    from tests._gpu import run_and_compare

    wl = wlm.WORKLOADS[wid]
    tally = run_and_compare(wl, wl.n_tokens, sample=_sample(wl.n_states, 6, wid), chunk=64)
    assert tally.entries > 0 and tally.worst_o <= 1e-4


def test_kda_workload_full_batch_one_window():
    """All 49,152 KDA head-states (24 layers x 32 heads x batch 64) for one window and a bit."""
    from tests._gpu import run_and_compare

    wl = wlm.WORKLOADS[5]
    run_and_compare(wl, wl.W + 4, sample=_sample(wl.n_states, 5, 55), chunk=wl.W + 4)


def test_kda_workload_full_length_requests_0_to_3():
    """Requests 0-3 of the KDA workload (all 24 x 32 layer-heads each: 3,072 head-states)
    over the full 2,048 tokens."""
    from tests._gpu import run_and_compare

    full = wlm.WORKLOADS[5]
    n = 4 * full.layers * full.heads
    wl = wlm.Workload(full.wid, full.name, n, full.n_tokens, True, "t3", full.n_warm, False, 4, full.layers,
                      full.heads)
    run_and_compare(wl, wl.n_tokens, sample=_sample(n, 4, 56), chunk=64)
