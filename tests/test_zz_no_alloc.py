"""lq_decode_step_noalloc: the mixed-phase decode step for callers that cannot allocate
device memory (an engine that owns all device memory and hands each part of the model
fixed buffers). Its work list lives in a fixed array of the library's device image
instead of the state buffer's work-list plane. The GPU test runs it and the ordinary
mixed-phase step (lq_decode_step with LQ_PHASE_ANY) on copies of one state whose
head-states sit at different window phases, for two calls in a row, each of which
fills some windows, and holds the outputs to the parity tolerance and the states to
bit equality. This file is collected last on purpose."""
import numpy as np
import pytest

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm


def test_noalloc_rejects_what_its_fixed_list_cannot_hold():
    lq.load()
    cfg = lq.config(window=4, n_comp=2)
    with pytest.raises(lq.LQError) as e:
        lq.decode_step_noalloc(cfg, 256, 65537, 256, 256, 256, 256, 256, 256, stream=0)
    assert e.value.code == lq.ERR_INVALID_ARG and "65536" in str(e.value)
    with pytest.raises(lq.LQError) as e:
        lq.decode_step_noalloc(lq.config(code_bits=4), 256, 8, 256, 256, 256, 256, 256, 256, stream=0)
    assert e.value.code == lq.ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("kda", [False, True])
def test_noalloc_matches_mixed_phase_step(kda):
    import torch

    from tests._gpu import to_dev
    from tests._helpers import rel_l2

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    N, W = 37, 4
    wl = wlm.custom(700 + kda, N, 0, kda=kda, n_warm=24, plant=True)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, 5)
    cfg = lq.config(window=W, n_comp=2, kda=kda)
    a = lq.alloc_state(cfg, N, dev)
    b = lq.alloc_state(cfg, N, dev)
    oa = torch.empty((N, 128), dtype=torch.float32, device=dev)
    ob = torch.empty_like(oa)
    # both copies reach the same mixed phases through the ordinary path: head-states
    # 10..19 are re-admitted before token 1 and 20..29 before token 2
    for st in (a, b):
        lq.state_init(cfg, st, N, to_dev(S0))
    for t in range(3):
        if t > 0:
            lo = 10 * t
            for st in (a, b):
                lq.state_init_range(cfg, st, N, lo, 10, to_dev(S0[lo:lo + 10]))
        for st, o in ((a, oa), (b, ob)):
            lq.decode_step(cfg, st, N, *(to_dev(x) for x in tk.token(t)), o)
    counts = lq.state_views(cfg, b, N)["counts"].cpu().numpy()
    assert sorted(set(counts.tolist())) == [1, 2, 3]
    for t in (3, 4):  # two calls in a row; each fills the windows of some head-states
        x = [to_dev(v) for v in tk.token(t)]
        full_before = int((lq.state_views(cfg, b, N)["counts"] == W - 1).sum())
        assert full_before > 0
        lq.decode_step(cfg, a, N, *x, oa)
        lq.decode_step_noalloc(cfg, b, N, *x, ob)
        assert lq.get_status(a) == (lq.OK, -1) and lq.get_status(b) == (lq.OK, -1)
        err = rel_l2(ob.cpu().numpy(), oa.cpu().numpy())
        assert err.max() <= 1e-4, (t, float(err.max()))
        # the boundaries and counts are equal, and so are the records each window holds
        # (record slots past a head-state's count hold nothing either call defined)
        va, vb = lq.state_views(cfg, a, N), lq.state_views(cfg, b, N)
        for name in ("counts", "codes", "sigma", "lambda", "comp_id", "comp_line"):
            assert torch.equal(va[name], vb[name]), (t, name)
        cnt = va["counts"].cpu().numpy()
        ra = va["rec_alpha"].view(N, W, -1)[:, :, :128] if kda else va["rec_alpha"][:, :W, None]
        rb = vb["rec_alpha"].view(N, W, -1)[:, :, :128] if kda else vb["rec_alpha"][:, :W, None]
        for st_i in range(N):
            held = int(cnt[st_i])
            for name in ("rec_k", "rec_u"):
                assert torch.equal(va[name][st_i, :held], vb[name][st_i, :held]), (t, name, st_i)
            assert torch.equal(ra[st_i, :held], rb[st_i, :held]), (t, "rec_alpha", st_i)
        assert int((lq.state_views(cfg, b, N)["counts"] == 0).sum()) >= full_before
