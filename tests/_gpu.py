"""GPU-side test harness: drives liblq through the binding and compares with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import FoldDiag, OracleState
from quantized_linear_attention_gb300 import lq
from quantized_linear_attention_gb300 import workload as wlm
from tests._helpers import near_tie, rel_l2

DEV = torch.device("cuda:0")


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV, non_blocking=False)


def unpack_codes(codes):
    """Code values (int8) from the codes plane: as is for 8-bit codes; 4-bit codes
    are two per byte (low nibble first), each stored as c + 8; 6-bit codes (96-byte
    rows) are stored as c + 32, low nibbles as a 4-bit row, then the top two bits of
    element e of block j at bits 8b + 2g of word j (g = 2(e//8) + e%2, b = (e%8)//2)."""
    if codes.dtype == np.int8:
        return codes
    if codes.shape[-1] == 96:
        nib = codes[..., :64]
        val = np.empty(codes.shape[:-1] + (128,), np.int16)
        val[..., 0::2] = nib & 0x0F
        val[..., 1::2] = nib >> 4
        hw = codes[..., 64:].copy().view("<u4")  # [..., 16-code block j]
        e = np.arange(16)
        shift = 8 * ((e % 8) // 2) + 2 * (2 * (e // 8) + e % 2)
        top = (hw[..., :, None] >> shift) & 3  # [..., j, e]
        val += (top.reshape(val.shape) << 4).astype(np.int16)
        return (val - 32).astype(np.int8)
    lo = (codes & 0x0F).astype(np.int16) - 8
    hi = (codes >> 4).astype(np.int16) - 8
    out = np.empty(codes.shape[:-1] + (2 * codes.shape[-1],), np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


class GpuState:
    def __init__(self, n, W=16, C=4, kda=False, smooth=True, lambda_floor=1e-6, code_bits=8, comp_fit=0,
                 comp_block=0):
        self.n, self.W, self.C, self.kda = n, W, C, kda
        self.cfg = lq.config(window=W, n_comp=C, kda=kda, smooth=smooth, lambda_floor=lambda_floor,
                             code_bits=code_bits, comp_fit=comp_fit, comp_block=comp_block)
        self.state = lq.alloc_state(self.cfg, n, DEV)
        self.views = lq.state_views(self.cfg, self.state, n)
        self.o = torch.empty((n, 128), dtype=torch.float32, device=DEV)

    def init(self, S0=None):
        lq.state_init(self.cfg, self.state, self.n, None if S0 is None else to_dev(S0))

    def step(self, q, k, v, a, b, phase=lq.PHASE_ANY):
        lq.decode_step(self.cfg, self.state, self.n, q, k, v, a, b, self.o, phase=phase)
        return self.o

    def append(self, q, k, v, a, b):
        lq.append(self.cfg, self.state, self.n, q, k, v, a, b, self.o)
        return self.o

    def fold(self):
        lq.fold(self.cfg, self.state, self.n)

    def export(self, idx=None):
        out = torch.empty((self.n, 128, 128), dtype=torch.float32, device=DEV)
        lq.export_state(self.cfg, self.state, self.n, out)
        if idx is not None:
            out = out.index_select(0, torch.as_tensor(list(idx), device=DEV))
        return out.cpu().numpy()

    def boundary(self, idx=None):
        idx = slice(None) if idx is None else torch.as_tensor(idx, device=DEV)
        v = self.views
        return dict(codes=unpack_codes(v["codes"][idx].cpu().numpy()), sigma=v["sigma"][idx].cpu().numpy(),
                    lam=v["lambda"][idx].cpu().numpy(), comp_id=v["comp_id"][idx].cpu().numpy(),
                    comp_line=v["comp_line"][idx].cpu().numpy(), count=v["counts"][idx].cpu().numpy())

    def status(self):
        return lq.get_status(self.state)


class Tally:
    """Codes compared so far and the mismatches allowed by the near-tie rule."""

    def __init__(self):
        self.entries = 0
        self.mismatch = 0
        self.worst_o = 0.0

    def check(self):
        assert self.mismatch <= 1e-5 * max(self.entries, 1), (self.mismatch, self.entries)


def compare_boundary(g, ref: OracleState, ref_idx, diags=None, tally: Tally | None = None, what=""):
    """GPU boundary dict g (states in the order of ref_idx) vs the oracle's states ref_idx."""
    C = ref.C
    ref_idx = list(ref_idx)
    assert np.array_equal(g["count"], ref.count[ref_idx]), what
    assert np.array_equal(g["comp_id"][:, :C], ref.comp_id[ref_idx, :C]), (what, g["comp_id"], ref.comp_id[ref_idx])
    # sigma, lambda and the compensator lines do not depend on how a tie rounds:
    # they are compared on every fold, whatever the codes do
    assert np.array_equal(g["sigma"], ref.sigma[ref_idx]), what
    assert np.array_equal(g["lam"], ref.lam[ref_idx]), what
    assert np.array_equal(g["comp_line"][:, :C], ref.comp_line[ref_idx, :C]), what
    codes_r = ref.codes[ref_idx]
    diff = g["codes"] != codes_r
    n = int(diff.sum())
    if tally is not None:
        tally.entries += codes_r.size
    if n:
        assert diags is not None, f"{what}: {n} code mismatches"
        s = np.stack([diags[i].s_round for i in range(len(ref_idx))])
        assert np.all(near_tie(s[diff])), f"{what}: {n} mismatches not at a tie"
        assert np.all(np.abs(g["codes"][diff].astype(int) - codes_r[diff]) <= 1), what
        if tally is not None:
            tally.mismatch += n
        return n
    return 0


def run_and_compare(wl: wlm.Workload, n_tokens: int, sample=None, phase_mode="stated", chunk=64, W=None, C=None,
                    smooth=True, tally=None, use_append_fold=False, code_bits=8, comp_fit=0, comp_block=0,
                    scale=1.0):
    """Free-running decode of n_tokens for all wl.n_states head-states on the GPU; the
    oracle follows the sampled states. Compares o every token, records every
    token, boundaries after every fold. `scale` (a power of two) multiplies the
    initial state and every v on both sides. Returns the Tally."""
    W = wl.W if W is None else W
    C = wl.C if C is None else C
    N = wl.n_states
    sample = list(range(N)) if sample is None else list(sample)
    tally = tally or Tally()
    S0, _ = wlm.initial_state(wl)
    sc = np.float32(scale)
    if S0 is not None and scale != 1.0:
        S0 = S0 * sc
    gpu = GpuState(N, W=W, C=C, kda=wl.kda, smooth=smooth, code_bits=code_bits, comp_fit=comp_fit,
                   comp_block=comp_block)
    gpu.init(S0)
    ref = OracleState(len(sample), W=W, C=C, decay_per_key=wl.kda, smooth=smooth, code_bits=code_bits,
                      comp_fit=comp_fit, comp_block=comp_block)
    d0 = [FoldDiag(128, 128) for _ in sample]
    ref.init(None if S0 is None else S0[sample], diags=d0)
    sidx = torch.as_tensor(sample, device=DEV)
    compare_boundary(gpu.boundary(sample), ref, range(len(sample)), d0, tally, "init")
    t = 0
    while t < n_tokens:
        n = min(chunk, n_tokens - t)
        tk = wlm.tokens(wl, t, n)
        if scale != 1.0:
            tk.v = tk.v * sc
        dq, dk, dv, da, db = (to_dev(x) for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta))
        sub = tk.select_states(sample)
        o_hist = torch.empty((n, len(sample), 128), dtype=torch.float32, device=DEV)
        for e in range(n):
            tt = t + e
            phase = tt % W if phase_mode == "stated" else lq.PHASE_ANY
            if use_append_fold:
                gpu.append(dq[e], dk[e], dv[e], da[e], db[e])
                if (tt + 1) % W == 0:
                    gpu.fold()
            else:
                gpu.step(dq[e], dk[e], dv[e], da[e], db[e], phase=phase)
            o_hist[e] = gpu.o.index_select(0, sidx)
            fills = (tt + 1) % W == 0
            o_ref = ref.run(*(x[e:e + 1] for x in (sub.q, sub.k, sub.v, sub.alpha, sub.beta)),
                            fold_when_full=False)[0]
            slot = tt % W
            g_u = gpu.views["rec_u"].index_select(0, sidx)[:, slot].cpu().numpy()
            assert np.array_equal(g_u, ref.rec_u[:, slot]), f"record u at token {tt}"
            # in units of the scale (exact in float64), so that the 1e-6 floor of the
            # relative error does not excuse outputs the scale made tiny
            err = rel_l2(o_hist[e].cpu().numpy().astype(np.float64) / scale, np.asarray(o_ref, np.float64) / scale)
            tally.worst_o = max(tally.worst_o, float(err.max()))
            assert err.max() <= 1e-4, (tt, err.max())
            if fills:
                dg = [FoldDiag(128, 128) for _ in sample]
                ref.fold(diags=dg)
                compare_boundary(gpu.boundary(sample), ref, range(len(sample)), dg, tally, f"fold at token {tt}")
        t += n
    st, bad = gpu.status()
    assert st == lq.OK, (lq.STATUS_NAMES.get(st), bad)
    # the state each head-state stands for, through lq_export_state
    ex = gpu.export(sample)
    ex_ref = ref.export()
    assert np.array_equal(ex, ex_ref)
    tally.check()
    return tally
