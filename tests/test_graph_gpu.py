"""lq_decode_step captured in a CUDA graph replays the same results as direct launches."""
import numpy as np
import pytest
import torch

from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_graph_replay_matches_direct_launches():
    wl = wlm.custom(600, 40, 0, n_warm=32, plant=True)
    S0, _ = wlm.initial_state(wl)
    tk = wlm.tokens(wl, 0, 16)
    dev_in = [torch.from_numpy(np.ascontiguousarray(x)).to(DEV) for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta)]
    cfg = lq.config()
    outs = []
    for use_graph in (False, True):
        # zero-filled so that padding bytes the library never writes compare equal
        st = torch.zeros(lq.state_bytes(cfg, 40), dtype=torch.uint8, device=DEV)
        lq.state_init(cfg, st, 40, torch.from_numpy(S0).to(DEV))
        o = torch.zeros(16, 40, 128, device=DEV)

        def window():
            for p in range(16):
                lq.decode_step(cfg, st, 40, *(x[p] for x in dev_in), o[p], phase=p)

        if use_graph:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
                window()
            g.replay()
        else:
            window()
        torch.cuda.synchronize()
        assert lq.get_status(st)[0] == lq.OK
        outs.append((o.cpu().numpy(), st.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
