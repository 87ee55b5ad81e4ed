"""Seeded synthetic workloads (inputs only) for per-window int8 decode.

Both the CUDA path and the CPU oracle are fed from this module, byte for byte.
It holds none of the quantization method's arithmetic: it draws per-token
q, k, v, alpha, beta and builds the fp32 initial state S0 (plain delta-rule
warm-up plus planted outlier lines). The generator itself is C
(``csrc/workload_gen.c``, counter-based SplitMix64), threaded over states.

The workloads are one Gated DeltaNet / KDA linear-attention layer shaped like
Qwen3.5-9B's (32 heads, one 128x128 state per head; fastpathlabs.ai research
note 4, "Background"), at the batch sizes that note times (32 / 128 / 512
requests, "Speed" table) plus a tiny case and a KDA case; see ``WORKLOADS``.
No dataset is involved: the note's recorded traces are not available, so these
seeded draws stand in for them with the same head shape and token count.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np

from . import build as _build

SEED = 0

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build_workload()
        L = ctypes.CDLL(path)
        u64, i64, i32, P = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.wl_tokens.restype = None
        L.wl_tokens.argtypes = [u64, u64, i32, i32, i32, i32, i64, i64, i64, i64, P, P, P, P, P, i32]
        L.wl_initial_state.restype = None
        L.wl_initial_state.argtypes = [u64, u64, i32, i32, i32, i32, i64, i64, i32, i32, P, P, i32]
        L.wl_raw_value.restype = u64
        L.wl_raw_value.argtypes = [u64] * 6
        L.wl_normal_value.restype = ctypes.c_double
        L.wl_normal_value.argtypes = [u64] * 6
        L.wl_mix64_value.restype = u64
        L.wl_mix64_value.argtypes = [u64]
        _lib = L
    return _lib


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (all states share d_k = d_v = 128, W = 16, C = 4)."""

    wid: int
    name: str
    n_states: int
    n_tokens: int
    kda: bool  # per-key-channel decay (KDA) instead of one scalar per token (GDN)
    vdist: str  # "normal" or "t3"
    n_warm: int  # plain delta-rule warm-up tokens before the init-fold
    plant: bool  # scale two rows and two columns of S0 by 30
    requests: int
    layers: int
    heads: int
    dk: int = 128
    dv: int = 128
    W: int = 16
    C: int = 4

    @property
    def vdist_id(self) -> int:
        return 1 if self.vdist == "t3" else 0

    @property
    def alpha_len(self) -> int:
        return self.dk if self.kda else 1

    def state_index(self, request, layer, head):
        return (request * self.layers + layer) * self.heads + head


WORKLOADS = {
    1: Workload(1, "gdn-tiny-1x2", 2, 64, False, "normal", 0, False, 1, 1, 2),
    2: Workload(2, "gdn-qwen3.5-9b-layer-batch32", 1024, 4095, False, "normal", 512, True, 32, 1, 32),
    3: Workload(3, "gdn-qwen3.5-9b-layer-batch128", 4096, 1024, False, "normal", 512, True, 128, 1, 32),
    4: Workload(4, "gdn-qwen3.5-9b-layer-batch512", 16384, 256, False, "normal", 512, True, 512, 1, 32),
    5: Workload(5, "kda-24x32-batch64", 49152, 2048, True, "t3", 512, False, 64, 24, 32),
}


def _ptr(a):
    return None if a is None else a.ctypes.data


def _threads(n):
    return int(n or os.cpu_count() or 1)


@dataclasses.dataclass
class Tokens:
    """Token-major inputs: q, k [T][N][dk]; v [T][N][dv]; alpha [T][N] or [T][N][dk]; beta [T][N]."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray

    def select_states(self, idx):
        return Tokens(self.q[:, idx], self.k[:, idx], self.v[:, idx], self.alpha[:, idx], self.beta[:, idx])

    def token(self, t):
        return self.q[t], self.k[t], self.v[t], self.alpha[t], self.beta[t]


def tokens(wl: Workload, tok0: int, n_tok: int, state0: int = 0, n_states: int | None = None, nthreads=None,
           states=None) -> Tokens:
    """Inputs for tokens [tok0, tok0+n_tok) of states [state0, state0+n_states) (or an explicit list)."""
    if states is not None:
        parts = [tokens(wl, tok0, n_tok, int(s), 1, nthreads=1) for s in states]
        return Tokens(*(np.concatenate([getattr(p, f) for p in parts], axis=1)
                        for f in ("q", "k", "v", "alpha", "beta")))
    N = wl.n_states - state0 if n_states is None else int(n_states)
    q = np.empty((n_tok, N, wl.dk), np.float32)
    k = np.empty((n_tok, N, wl.dk), np.float32)
    v = np.empty((n_tok, N, wl.dv), np.float32)
    alpha = np.empty((n_tok, N, wl.dk) if wl.kda else (n_tok, N), np.float32)
    beta = np.empty((n_tok, N), np.float32)
    _load().wl_tokens(SEED, wl.wid, int(wl.kda), wl.vdist_id, wl.dk, wl.dv, state0, N, tok0, n_tok, _ptr(q),
                      _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _threads(nthreads))
    return Tokens(q, k, v, alpha, beta)


def initial_state(wl: Workload, state0: int = 0, n_states: int | None = None, nthreads=None, states=None):
    """(S0 [N][dv][dk] fp32, planted [N][4] int32) -- None, None when the workload starts from zero."""
    if wl.n_warm == 0 and not wl.plant:
        return None, None
    if states is not None:
        parts = [initial_state(wl, int(s), 1, nthreads=1) for s in states]
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])
    N = wl.n_states - state0 if n_states is None else int(n_states)
    S0 = np.empty((N, wl.dv, wl.dk), np.float32)
    planted = np.empty((N, 4), np.int32)
    _load().wl_initial_state(SEED, wl.wid, int(wl.kda), wl.vdist_id, wl.dk, wl.dv, state0, N, wl.n_warm,
                             int(wl.plant), _ptr(S0), _ptr(planted), _threads(nthreads))
    return S0, planted


def raw_value(wid, state, token, tensor, e):
    return int(_load().wl_raw_value(SEED, wid, state, token, tensor, e))


def mix64(z):
    return int(_load().wl_mix64_value(z))


def normal_value(wid, state, token, tensor, e):
    return float(_load().wl_normal_value(SEED, wid, state, token, tensor, e))


def custom(wid: int, n_states: int, n_tokens: int, kda=False, vdist="normal", n_warm=0, plant=False, **kw):
    """An ad-hoc workload (for edge cases: ragged or tiny batches) with its own stream id."""
    return Workload(wid, f"custom-{wid}", n_states, n_tokens, kda, vdist, n_warm, plant, 1, 1, n_states, **kw)
