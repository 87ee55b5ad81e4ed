"""Thin Python binding of ``liblq.so`` (C ABI in ``include/lq.h``).

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels. Tensors are torch CUDA tensors (PyTorch supplies device memory
and streams); each call passes their device pointers and the current (or
given) CUDA stream. The library is loaded on first use; if it is missing the
call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

PHASE_ANY = -1

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WINDOW_FULL = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5
ERR_PHASE = -6
ERR_STATE = -7

STATUS_NAMES = {0: "LQ_OK", -1: "LQ_ERR_INVALID_ARG", -2: "LQ_ERR_UNSUPPORTED", -3: "LQ_ERR_WINDOW_FULL",
                -4: "LQ_ERR_CUDA", -5: "LQ_ERR_TIMEOUT", -6: "LQ_ERR_PHASE", -7: "LQ_ERR_STATE"}

# Every symbol include/lq.h declares.
EXPORTS = ("lq_config_default", "lq_state_bytes", "lq_layout", "lq_state_init", "lq_state_init_range", "lq_append",
           "lq_fold", "lq_decode_step", "lq_decode_step_noalloc", "lq_decode_step2", "lq_decode_step_rwkv7", "lq_export_state",
           "lq_fp32_decode_step", "lq_get_status", "lq_clear_status", "lq_last_error", "lq_version",
           "lq_debug_set_wait")


class Config(ctypes.Structure):
    _fields_ = [("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("window", ctypes.c_int32),
                ("n_comp", ctypes.c_int32), ("decay_per_key", ctypes.c_int32), ("smooth", ctypes.c_int32),
                ("lambda_floor", ctypes.c_float), ("code_bits", ctypes.c_int32), ("comp_fit", ctypes.c_int32),
                ("comp_block", ctypes.c_int32)]


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("total_bytes", "header", "counts", "codes", "sigma", "lambda_",
                                                "comp_id", "comp_line", "rec_k", "rec_u", "rec_alpha",
                                                "full_list")] + \
               [("comp_id_stride", ctypes.c_int64), ("alpha_stride", ctypes.c_int64),
                ("boundary_bytes_per_state", ctypes.c_int64)]


class LQError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def library_path() -> str:
    return _build.lq_library_path()


def load():
    """Load liblq.so (built in-tree by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"liblq.so not found at {path}: build it first (python -c 'import __graft_entry__ as g; "
                           f"g.build()'); there is no fallback path")
    L = ctypes.CDLL(path)
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    cfgp = ctypes.POINTER(Config)
    sig = {
        "lq_config_default": (None, [cfgp]),
        "lq_state_bytes": (ctypes.c_size_t, [cfgp, i64]),
        "lq_layout": (ctypes.c_int, [cfgp, i64, ctypes.POINTER(Layout)]),
        "lq_state_init": (ctypes.c_int, [cfgp, P, i64, P, P]),
        "lq_state_init_range": (ctypes.c_int, [cfgp, P, i64, i64, i64, P, P]),
        "lq_append": (ctypes.c_int, [cfgp, P, i64, P, P, P, P, P, P, P]),
        "lq_fold": (ctypes.c_int, [cfgp, P, i64, P]),
        "lq_decode_step": (ctypes.c_int, [cfgp, P, i64, i32, P, P, P, P, P, P, P]),
        "lq_decode_step_noalloc": (ctypes.c_int, [cfgp, P, i64, P, P, P, P, P, P, P]),
        "lq_decode_step2": (ctypes.c_int, [cfgp, P, i64, i32, P, P, P, P, P, P, P, P, P, P]),
        "lq_decode_step_rwkv7": (ctypes.c_int, [cfgp, P, i64, i32, P, P, P, P, P, P, P, P]),
        "lq_export_state": (ctypes.c_int, [cfgp, P, i64, P, P]),
        "lq_fp32_decode_step": (ctypes.c_int, [cfgp, P, i64, P, P, P, P, P, P, P]),
        "lq_get_status": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_int64), P]),
        "lq_clear_status": (ctypes.c_int, [P, P]),
        "lq_last_error": (ctypes.c_char_p, []),
        "lq_version": (ctypes.c_int, []),
        "lq_debug_set_wait": (ctypes.c_int, [ctypes.c_uint64, i32, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def last_error() -> str:
    return load().lq_last_error().decode()


def _check(rc):
    if rc != OK:
        raise LQError(rc, last_error())


def config(window=16, n_comp=4, kda=False, smooth=True, lambda_floor=1e-6, d_k=128, d_v=128, code_bits=8,
           comp_fit=0, comp_block=0) -> Config:
    return Config(d_k, d_v, window, n_comp, int(bool(kda)), int(bool(smooth)), lambda_floor, code_bits, comp_fit,
                  int(comp_block))


def default_config() -> Config:
    c = Config()
    load().lq_config_default(ctypes.byref(c))
    return c


def state_bytes(cfg: Config, n_states: int) -> int:
    return int(load().lq_state_bytes(ctypes.byref(cfg), n_states))


def layout(cfg: Config, n_states: int) -> Layout:
    out = Layout()
    _check(load().lq_layout(ctypes.byref(cfg), n_states, ctypes.byref(out)))
    return out


# ---------------------------------------------------------------------------- marshalling
def _ptr(t, name, dtype=None):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    import torch

    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _f32():
    import torch

    return torch.float32


def alloc_state(cfg: Config, n_states: int, device="cuda"):
    """Caller-owned state buffer (torch supplies the memory)."""
    import torch

    return torch.empty(state_bytes(cfg, n_states), dtype=torch.uint8, device=device)


def state_init(cfg, state, n_states, S0=None, stream=None):
    _check(load().lq_state_init(ctypes.byref(cfg), _ptr(state, "state"), n_states, _ptr(S0, "S0", _f32()),
                                _stream(stream)))


def state_init_range(cfg, state, n_states, first, count, S0=None, stream=None):
    """Re-initialise head-states first .. first+count-1 from S0 [count][d_v][d_k] (None: zero)."""
    _check(load().lq_state_init_range(ctypes.byref(cfg), _ptr(state, "state"), n_states, int(first), int(count),
                                      _ptr(S0, "S0", _f32()), _stream(stream)))


def append(cfg, state, n_states, q, k, v, alpha, beta, o, stream=None):
    f = _f32()
    _check(load().lq_append(ctypes.byref(cfg), _ptr(state, "state"), n_states, _ptr(q, "q", f), _ptr(k, "k", f),
                            _ptr(v, "v", f), _ptr(alpha, "alpha", f), _ptr(beta, "beta", f), _ptr(o, "o", f),
                            _stream(stream)))


def fold(cfg, state, n_states, stream=None):
    _check(load().lq_fold(ctypes.byref(cfg), _ptr(state, "state"), n_states, _stream(stream)))


def decode_step(cfg, state, n_states, q, k, v, alpha, beta, o, phase=PHASE_ANY, stream=None):
    f = _f32()
    _check(load().lq_decode_step(ctypes.byref(cfg), _ptr(state, "state"), n_states, int(phase), _ptr(q, "q", f),
                                 _ptr(k, "k", f), _ptr(v, "v", f), _ptr(alpha, "alpha", f), _ptr(beta, "beta", f),
                                 _ptr(o, "o", f), _stream(stream)))


def decode_step_noalloc(cfg, state, n_states, q, k, v, alpha, beta, o, stream=None):
    """Mixed-phase decode step whose work list lives in the library's fixed device array
    (for callers that cannot allocate device memory); arguments as ``decode_step``."""
    f = _f32()
    _check(load().lq_decode_step_noalloc(ctypes.byref(cfg), _ptr(state, "state"), n_states, _ptr(q, "q", f),
                                         _ptr(k, "k", f), _ptr(v, "v", f), _ptr(alpha, "alpha", f),
                                         _ptr(beta, "beta", f), _ptr(o, "o", f), _stream(stream)))


def decode_step2(cfg, state, n_states, q, k1, v1, beta1, k2, v2, beta2, alpha, o, phase=PHASE_ANY, stream=None):
    """One two-record token (records (k1, u1, alpha) and (k2, u2, 1)); o = S_{n+1} q."""
    f = _f32()
    _check(load().lq_decode_step2(ctypes.byref(cfg), _ptr(state, "state"), n_states, int(phase), _ptr(q, "q", f),
                                  _ptr(k1, "k1", f), _ptr(v1, "v1", f), _ptr(beta1, "beta1", f), _ptr(k2, "k2", f),
                                  _ptr(v2, "v2", f), _ptr(beta2, "beta2", f), _ptr(alpha, "alpha", f),
                                  _ptr(o, "o", f), _stream(stream)))


def decode_step_rwkv7(cfg, state, n_states, r, w, kh, a, k, v, o, phase=PHASE_ANY, stream=None):
    """One RWKV7 token: the erase record (a . kh, -(S kh), w), then the pure write (k, v, 1); o = S r."""
    f = _f32()
    _check(load().lq_decode_step_rwkv7(ctypes.byref(cfg), _ptr(state, "state"), n_states, int(phase),
                                       _ptr(r, "r", f), _ptr(w, "w", f), _ptr(kh, "kh", f), _ptr(a, "a", f),
                                       _ptr(k, "k", f), _ptr(v, "v", f), _ptr(o, "o", f), _stream(stream)))


def export_state(cfg, state, n_states, S_out, stream=None):
    _check(load().lq_export_state(ctypes.byref(cfg), _ptr(state, "state"), n_states, _ptr(S_out, "S_out", _f32()),
                                  _stream(stream)))


def fp32_decode_step(cfg, S, n_states, q, k, v, alpha, beta, o, stream=None):
    """The fp32-state baseline: one plain delta-rule token on whole fp32 states S [n][d_v][d_k], in place."""
    f = _f32()
    _check(load().lq_fp32_decode_step(ctypes.byref(cfg), _ptr(S, "S", f), n_states, _ptr(q, "q", f), _ptr(k, "k", f),
                                      _ptr(v, "v", f), _ptr(alpha, "alpha", f), _ptr(beta, "beta", f),
                                      _ptr(o, "o", f), _stream(stream)))


def get_status(state, stream=None):
    """(status, bad_state): synchronizes the stream and reads the device status word."""
    bad = ctypes.c_int64(-1)
    rc = load().lq_get_status(_ptr(state, "state"), ctypes.byref(bad), _stream(stream))
    if rc in (ERR_INVALID_ARG, ERR_CUDA):
        raise LQError(rc, last_error())
    return rc, bad.value


def clear_status(state, stream=None):
    _check(load().lq_clear_status(_ptr(state, "state"), _stream(stream)))


def debug_set_wait(wait_ns=0, extra_tx_append=0, extra_tx_fold=0):
    """Test hook: this thread's bound on kernel waits and the bytes the append / fold
    kernels announce beyond those they copy (so the wait runs out). (0, 0, 0) restores
    the defaults."""
    _check(load().lq_debug_set_wait(int(wait_ns), int(extra_tx_append), int(extra_tx_fold)))


def state_views(cfg: Config, state, n_states: int) -> dict:
    """Typed torch views of the planes of a state buffer (no copy), per ``lq_layout``. With
    4- or 6-bit codes, "codes" is the packed plane, uint8 [N][d_v][d_k * bits / 8]
    (the layout ``include/lq.h`` gives)."""
    import torch

    L = layout(cfg, n_states)
    N, D, W, C = n_states, cfg.d_k, cfg.window, cfg.n_comp

    def view(off, count, dtype, shape):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return state[off:off + nbytes].view(dtype).view(*shape)

    return {
        "counts": view(L.counts, N, torch.int32, (N,)),
        "codes": (view(L.codes, N * D * D, torch.int8, (N, D, D)) if cfg.code_bits == 8 else
                  view(L.codes, N * D * D * cfg.code_bits // 8, torch.uint8, (N, D, D * cfg.code_bits // 8))),
        "sigma": view(L.sigma, N * D, torch.float32, (N, D)),
        "lambda": view(L.lambda_, N * D, torch.float32, (N, D)),
        "comp_id": view(L.comp_id, N * L.comp_id_stride, torch.int32, (N, L.comp_id_stride))[:, :C],
        "comp_line": view(L.comp_line, N * C * D * (2 if cfg.comp_fit else 1), torch.float32,
                          (N, C, D * (2 if cfg.comp_fit else 1))),
        "rec_k": view(L.rec_k, N * W * D, torch.float32, (N, W, D)),
        "rec_u": view(L.rec_u, N * W * D, torch.float32, (N, W, D)),
        "rec_alpha": view(L.rec_alpha, N * L.alpha_stride, torch.float32, (N, L.alpha_stride)),
        "full_list": view(L.full_list, N, torch.int32, (N,)),
    }
