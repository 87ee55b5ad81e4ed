"""Python front of the CPU oracle (``lq_oracle.c``).

TEST INFRASTRUCTURE, NOT THE PRODUCT: only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg and reference arm may import this module. It loads the oracle's
own C library (built from ``oracle/lq_oracle.c`` by ``oracle/build.py``) and holds
per-state arrays in numpy. No code here is shared with the CUDA path.

The arithmetic lives in C; this file only owns memory and marshals pointers.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class Cfg(ctypes.Structure):
    _fields_ = [
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("W", ctypes.c_int32),
        ("C", ctypes.c_int32),
        ("decay_per_key", ctypes.c_int32),
        ("smooth", ctypes.c_int32),
        ("quantize", ctypes.c_int32),
        ("lambda_floor", ctypes.c_float),
        ("code_bits", ctypes.c_int32),
        ("comp_fit", ctypes.c_int32),
        ("comp_block", ctypes.c_int32),
    ]


_P = ctypes.c_void_p


class Batch(ctypes.Structure):
    _fields_ = [
        ("n_states", ctypes.c_int64),
        ("codes", _P),
        ("sigma", _P),
        ("lambda_", _P),
        ("comp_id", _P),
        ("comp_line", _P),
        ("B", _P),
        ("rec_k", _P),
        ("rec_u", _P),
        ("rec_alpha", _P),
        ("count", _P),
    ]


class Diag(ctypes.Structure):
    _fields_ = [("S", _P), ("R", _P), ("s_round", _P)]


def lib():
    """Load (building if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.library_path()
        if not os.path.exists(path) or _build.stale():
            _build.build()
        L = ctypes.CDLL(path)
        L.orc_dot.restype = ctypes.c_float
        L.orc_dot.argtypes = [ctypes.c_int, _P, ctypes.c_long, _P, ctypes.c_long]
        L.orc_sum_abs.restype = ctypes.c_float
        L.orc_sum_abs.argtypes = [ctypes.c_int, _P, ctypes.c_long]
        for name in ("orc_init_state", "orc_append", "orc_fold", "orc_export", "orc_run"):
            getattr(L, name).restype = ctypes.c_int
        L.orc_init_state.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, _P,
                                     ctypes.POINTER(Diag)]
        L.orc_append.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, _P, _P, _P, _P,
                                 ctypes.c_float, _P]
        L.orc_fold.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, ctypes.POINTER(Diag)]
        L.orc_export.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, _P]
        L.orc_run.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, _P, _P, _P, _P, _P, _P,
                              ctypes.c_int, ctypes.c_int]
        L.orc_append_rwkv.restype = ctypes.c_int
        L.orc_append_rwkv.argtypes = [ctypes.POINTER(Cfg), ctypes.POINTER(Batch), ctypes.c_int64, _P, _P, _P, _P, _P,
                                      _P, _P]
        L.orc_fit.restype = ctypes.c_int
        L.orc_fit.argtypes = [ctypes.POINTER(Cfg), _P, _P, _P, _P]
        L.orc_fp32_run.restype = None
        L.orc_fp32_run.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _P,
                                   _P, _P, _P, _P, _P, _P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def dot(a, b) -> float:
    """The oracle's fixed-order dot product of two fp32 vectors."""
    a, b = _f32(a), _f32(b)
    assert a.shape == b.shape and a.ndim == 1
    return float(lib().orc_dot(a.size, _ptr(a), 1, _ptr(b), 1))


def sum_abs(a) -> float:
    a = _f32(a)
    return float(lib().orc_sum_abs(a.size, _ptr(a), 1))


class FoldDiag:
    """Per-state fold diagnostics: S before selection, residual R, pre-round values."""

    def __init__(self, dv, dk):
        self.S = np.zeros((dv, dk), np.float32)
        self.R = np.zeros((dv, dk), np.float32)
        self.s_round = np.zeros((dv, dk), np.float32)
        self.c = Diag(_ptr(self.S), _ptr(self.R), _ptr(self.s_round))


class OracleState:
    """Boundary + record buffer for ``n_states`` head-states, as numpy arrays."""

    def __init__(self, n_states, dk=128, dv=128, W=16, C=4, decay_per_key=False, smooth=True, quantize=True,
                 lambda_floor=1e-6, code_bits=8, comp_fit=0, comp_block=0):
        self.n, self.dk, self.dv, self.W, self.C = int(n_states), int(dk), int(dv), int(W), int(C)
        self.kda = bool(decay_per_key)
        self.code_bits = int(code_bits)
        self.comp_fit = int(comp_fit)
        self.comp_block = int(comp_block)
        self.cfg = Cfg(self.dk, self.dv, self.W, self.C, int(decay_per_key), int(smooth), int(quantize),
                       float(lambda_floor), self.code_bits, self.comp_fit, self.comp_block)
        N, L = self.n, max(self.dk, self.dv)
        alen = self.dk if self.kda else 1
        self.codes = np.zeros((N, self.dv, self.dk), np.int8)
        self.sigma = np.zeros((N, self.dv), np.float32)
        self.lam = np.ones((N, self.dk), np.float32)
        self.comp_id = np.zeros((N, max(self.C, 1)), np.int32)
        # one line per compensator, or with fitted factors a (d_v) then b (d_k)
        clen = self.dv + self.dk if self.comp_fit > 0 else L
        self.comp_line = np.zeros((N, max(self.C, 1), clen), np.float32)
        self.B = np.zeros((N, self.dv, self.dk), np.float32) if not quantize else None
        self.rec_k = np.zeros((N, self.W, self.dk), np.float32)
        self.rec_u = np.zeros((N, self.W, self.dv), np.float32)
        self.rec_alpha = np.zeros((N, self.W, alen), np.float32)
        self.count = np.zeros((N,), np.int32)
        self.batch = Batch(N, _ptr(self.codes), _ptr(self.sigma), _ptr(self.lam), _ptr(self.comp_id),
                           _ptr(self.comp_line), _ptr(self.B), _ptr(self.rec_k), _ptr(self.rec_u),
                           _ptr(self.rec_alpha), _ptr(self.count))

    # -- per-state calls -------------------------------------------------
    def init(self, S0=None, diags=None):
        """Init-fold every state from S0 [N][dv][dk] (None: zero)."""
        L = lib()
        if S0 is not None:
            S0 = _f32(S0).reshape(self.n, self.dv, self.dk)
        for s in range(self.n):
            p = None if S0 is None else S0[s].ctypes.data
            d = None if diags is None else ctypes.byref(diags[s].c)
            rc = L.orc_init_state(ctypes.byref(self.cfg), ctypes.byref(self.batch), s, p, d)
            if rc != 0:
                raise RuntimeError(f"orc_init_state failed: {rc}")

    def init_range(self, first, count, S0=None, diags=None):
        """Init-fold states first .. first+count-1 from S0 [count][dv][dk] (None: zero);
        the other states keep their boundaries and records."""
        L = lib()
        if S0 is not None:
            S0 = _f32(S0).reshape(count, self.dv, self.dk)
        for i in range(count):
            p = None if S0 is None else S0[i].ctypes.data
            d = None if diags is None else ctypes.byref(diags[i].c)
            rc = L.orc_init_state(ctypes.byref(self.cfg), ctypes.byref(self.batch), first + i, p, d)
            if rc != 0:
                raise RuntimeError(f"orc_init_state failed: {rc}")

    def append(self, q, k, v, alpha, beta):
        """Append one token to every state; returns o [N][dv] (float64)."""
        return self.run(np.asarray(q)[None], np.asarray(k)[None], np.asarray(v)[None], np.asarray(alpha)[None],
                        np.asarray(beta)[None], fold_when_full=False)[0]

    def fold(self, states=None, diags=None):
        L = lib()
        for idx, s in enumerate(range(self.n) if states is None else states):
            d = None if diags is None else ctypes.byref(diags[idx].c)
            rc = L.orc_fold(ctypes.byref(self.cfg), ctypes.byref(self.batch), int(s), d)
            if rc != 0:
                raise RuntimeError(f"orc_fold failed: {rc}")

    def export(self):
        """S_n [N][dv][dk]: the state the boundary plus records stand for."""
        out = np.zeros((self.n, self.dv, self.dk), np.float32)
        L = lib()
        for s in range(self.n):
            rc = L.orc_export(ctypes.byref(self.cfg), ctypes.byref(self.batch), s, out[s].ctypes.data)
            if rc != 0:
                raise RuntimeError(f"orc_export failed: {rc}")
        return out

    def run(self, q, k, v, alpha, beta, fold_when_full=True, nthreads=None, want_o=True):
        """Decode T tokens: q,k [T][N][dk], v [T][N][dv], alpha [T][N] or [T][N][dk], beta [T][N].

        Each token: append, then fold if the window is full (``fold_when_full``).
        Returns o [T][N][dv] in float64 (or None).
        """
        q, k, v, alpha, beta = (_f32(x) for x in (q, k, v, alpha, beta))
        T = q.shape[0]
        assert q.shape == (T, self.n, self.dk) and k.shape == q.shape and v.shape == (T, self.n, self.dv)
        assert alpha.size == T * self.n * (self.dk if self.kda else 1) and beta.size == T * self.n
        o = np.zeros((T, self.n, self.dv), np.float64) if want_o else None
        nthreads = nthreads or os.cpu_count() or 1
        rc = lib().orc_run(ctypes.byref(self.cfg), ctypes.byref(self.batch), T, _ptr(q), _ptr(k), _ptr(v),
                           _ptr(alpha), _ptr(beta), _ptr(o), int(bool(fold_when_full)), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"orc_run failed: {rc}")
        return o

    def append_rwkv(self, r, w, kh, a, k, v):
        """One RWKV7 token (erase record, then pure-write record) into every state:
        r, w, kh, a, k [N][dk], v [N][dv]. Returns o [N][dv] (float64)."""
        r, w, kh, a, k, v = (_f32(x) for x in (r, w, kh, a, k, v))
        o = np.zeros((self.n, self.dv), np.float64)
        L = lib()
        for s in range(self.n):
            rc = L.orc_append_rwkv(ctypes.byref(self.cfg), ctypes.byref(self.batch), s, _ptr(r[s]), _ptr(w[s]),
                                   _ptr(kh[s]), _ptr(a[s]), _ptr(k[s]), _ptr(v[s]), _ptr(o[s]))
            if rc != 0:
                raise RuntimeError(f"orc_append_rwkv failed: {rc}")
        return o

    # -- views -------------------------------------------------------------
    def boundary(self, s):
        """Boundary of state s as a dict of numpy copies."""
        d = dict(codes=self.codes[s].copy(), sigma=self.sigma[s].copy(), lam=self.lam[s].copy(),
                 comp_id=self.comp_id[s, :self.C].copy(), comp_line=self.comp_line[s, :self.C].copy(),
                 count=int(self.count[s]))
        return d

    def dequant(self, s):
        """B (fp64) of state s: Diag(sigma) Cd Diag(lambda) plus the compensator terms."""
        B = (self.sigma[s].astype(np.float64)[:, None] * self.codes[s].astype(np.float64)
             * self.lam[s].astype(np.float64)[None, :])
        for c in range(self.C):
            if self.comp_fit > 0:
                line = self.comp_line[s, c].astype(np.float64)
                B += np.outer(line[:self.dv], line[self.dv:])
                continue
            cid = int(self.comp_id[s, c])
            if cid < self.dv:
                B[cid, :] += self.comp_line[s, c, :self.dk]
            else:
                B[:, cid - self.dv] += self.comp_line[s, c, :self.dv]
        return B


def fit(R, C, sweeps, block=False, prev=None):
    """F2 alone on R [dv][dk] (fp32): returns (a [C][dv], b [C][dk], ids [C], the deflated
    residual). block: the block fit, from prev = (a, b) of the previous window when given."""
    R = _f32(R).copy()
    dv, dk = R.shape
    cfg = Cfg(dk, dv, 16, C, 0, 1, 1, 1e-6, 8, int(sweeps), int(bool(block)))
    out = np.zeros((C, dv + dk), np.float32)
    ids = np.zeros(C, np.int32)
    pl = None
    if prev is not None:
        pl = np.ascontiguousarray(np.concatenate([_f32(prev[0]), _f32(prev[1])], axis=1))
    rc = lib().orc_fit(ctypes.byref(cfg), _ptr(R), _ptr(pl), _ptr(out), _ptr(ids))
    if rc != 0:
        raise RuntimeError(f"orc_fit failed: {rc}")
    return out[:, :dv], out[:, dv:], ids, R


def fp32_run(S0, q, k, v, alpha, beta, want_o=True):
    """The fp32-state baseline recurrence (plain per-token delta rule, whole state),
    evaluated in double. S0 [n][d_v][d_k]; inputs token-major. Returns (S_T, o [T][n][d_v])."""
    q, k, v, alpha, beta = (_f32(x) for x in (q, k, v, alpha, beta))
    T, n, dk = q.shape
    dv = v.shape[2]
    S = np.ascontiguousarray(S0, dtype=np.float64).copy()
    o = np.empty((T, n, dv), np.float64) if want_o else None
    lib().orc_fp32_run(dk, dv, int(alpha.ndim == 3), n, T, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                       _ptr(o) if want_o else None)
    return S, o
