"""Seeded random sweep over the configuration space, against the oracle.

Each case draws a window length, compensator count, code width, decay form,
compensator form, head-state count, token form (one-record tokens at stated or
mixed phases, two-record tokens, RWKV7 tokens, staggered admissions) and an
input mix (normal or Student-t(3) values, warm-started or zero initial states,
planted outliers), then runs the matching parity harness. Every case holds the
harness's own bar: records and codes exact (codes except at rounding ties),
outputs within 1e-4 relative L2. Zero initial states make the first token's
output a single dot product k . q, which is where a float sum of the products
would lose digits.
"""
import random

import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._gpu import run_and_compare
from tests.test_parity_rwkv_gpu import run_rwkv
from tests.test_parity_stagger_gpu import _groups, run_staggered
from tests.test_parity_two_gpu import run_two

pytestmark = pytest.mark.gpu

CASES = 60


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lq.load()
    torch.cuda.set_device(0)


def _draw(rng, i):
    W = rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 24, 32])
    C = rng.randint(0, 8)
    bits = rng.choice([8, 8, 6, 4])
    kda = rng.random() < 0.4
    fit = rng.choice([0, 0, 0, 1, 2]) if C > 0 else 0
    block = rng.randint(0, 1) if fit else 0
    n = rng.choice([1, 2, 3, 7, 19, 40, 150])
    form = rng.choice(["one", "one", "any", "two", "rwkv", "stagger"])
    if form == "two" and W < 2:
        form = "one"
    if form == "rwkv" and (W < 2 or not kda):
        form = "one"
    if form == "stagger" and W < 2:
        form = "any"
    wl = wlm.custom(20000 + i, n, 0, kda=kda, vdist=rng.choice(["normal", "t3"]), n_warm=rng.choice([0, 16, 64]),
                    plant=rng.random() < 0.5)
    return dict(W=W, C=C, bits=bits, fit=fit, block=block, n=n, form=form, wl=wl)


def _run(rng, c, i):
    W, C, bits, fit, block, wl = c["W"], c["C"], c["bits"], c["fit"], c["block"], c["wl"]
    if c["form"] in ("one", "any"):
        run_and_compare(wl, rng.randint(W, 3 * W) if W > 1 else 5, W=W, C=C,
                        phase_mode="stated" if c["form"] == "one" else "any", code_bits=bits, comp_fit=fit,
                        comp_block=block)
    elif c["form"] == "two":
        n_tok = rng.randint(max(1, W // 2), 2 * W) if W % 2 == 0 else max(1, (W - 1) // 2)
        run_two(wl, n_tok, W=W, C=C, code_bits=bits, comp_fit=fit)
    elif c["form"] == "rwkv":
        n_tok = max(1, rng.randint(W // 2, 2 * W)) if W % 2 == 0 else max(1, (W - 1) // 2)
        run_rwkv(wl, n_tok, W=W, C=C, code_bits=bits, comp_fit=fit, comp_block=block)
    else:
        run_staggered(wl, rng.randint(W, 3 * W), _groups(c["n"], min(c["n"], W), i), W=W, C=C, code_bits=bits,
                      comp_fit=fit)


@pytest.mark.parametrize("seed", [5, 17])
def test_random_configurations(seed):
    rng = random.Random(seed)
    failed = []
    for i in range(CASES):
        c = _draw(rng, 1000 * seed + i)
        try:
            _run(rng, c, i)
        except AssertionError as e:
            desc = {k: v for k, v in c.items() if k != "wl"}
            failed.append(f"case {i} {desc}: {str(e)[:200]}")
    assert not failed, "\n".join(failed)
