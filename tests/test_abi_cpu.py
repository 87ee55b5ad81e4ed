"""The C-ABI library on the host (no GPU): symbols, layout, validation."""
import ctypes
import os
import re
import threading

import pytest

from quantized_linear_attention_gb300 import build as lq_build
from quantized_linear_attention_gb300 import lq
from tests._helpers import read_golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    lq_build.build_lq()
    return lq.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert names == sorted(lq.EXPORTS)
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {lq.library_path()}").read()
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_version_and_default(L):
    assert lq.load().lq_version() >= 100
    c = lq.default_config()
    assert (c.d_k, c.d_v, c.window, c.n_comp, c.decay_per_key, c.smooth) == (128, 128, 16, 4, 0, 1)
    assert abs(c.lambda_floor - 1e-6) < 1e-12


def test_pin8_boundary_bytes_per_element(L):
    """PIN-8: the boundary takes 1.19 bytes per state element (LeapQuant summary, §4.3)."""
    g = read_golden("page_figures.txt")
    lay = lq.layout(lq.default_config(), 1)
    per_elem = lay.boundary_bytes_per_state / (128 * 128)
    assert lay.boundary_bytes_per_state == 16384 + 512 + 512 + 4 * 4 + 4 * 512 == 19472
    assert round(per_elem, 2) == g["boundary_bytes_per_element"]
    assert round(4 / per_elem, 1) == g["boundary_storage_reduction"]


def test_boundary_bytes_with_4bit_codes(L):
    """4-bit codes (LeapQuant §4 also evaluates 4-bit states): two codes per byte,
    so the boundary takes 8192 + 512 + 512 + 4C + 512C bytes, 0.69 per element."""
    lay = lq.layout(lq.config(code_bits=4), 1)
    assert lay.boundary_bytes_per_state == 8192 + 512 + 512 + 4 * 4 + 4 * 512 == 11280
    assert round(lay.boundary_bytes_per_state / (128 * 128), 2) == 0.69
    l8 = lq.layout(lq.config(), 1000)
    l4 = lq.layout(lq.config(code_bits=4), 1000)
    assert l8.total_bytes - l4.total_bytes == 1000 * 8192
    assert l4.sigma - l4.codes == 1000 * 8192


def test_boundary_bytes_with_6bit_codes(L):
    """6-bit codes (LeapQuant §4 also evaluates 6-bit states): 96 bytes per row, so
    the boundary takes 12288 + 512 + 512 + 4C + 512C bytes, 0.94 per element."""
    lay = lq.layout(lq.config(code_bits=6), 1)
    assert lay.boundary_bytes_per_state == 12288 + 512 + 512 + 4 * 4 + 4 * 512 == 15376
    assert round(lay.boundary_bytes_per_state / (128 * 128), 2) == 0.94
    l6 = lq.layout(lq.config(code_bits=6), 1000)
    assert l6.sigma - l6.codes == 1000 * 12288


def test_fitted_factor_compensators_double_the_compensator_plane(L):
    """With comp_fit > 0 each compensator is a factor pair a (d_v) and b (d_k)."""
    l0 = lq.layout(lq.config(), 1)
    l1 = lq.layout(lq.config(comp_fit=8), 1)
    assert l1.boundary_bytes_per_state - l0.boundary_bytes_per_state == 4 * 4 * 128
    assert l0.rec_k - l0.comp_line == 4 * 4 * 128  # C = 4 lines of 128 floats (256-byte aligned already)
    assert l1.rec_k - l1.comp_line == 4 * 4 * 256  # C = 4 pairs of 128 + 128 floats
    assert l1.total_bytes - l0.total_bytes == 4 * 4 * 128


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("n", [1, 3, 1024, 16384])
def test_layout_planes(L, n, kda):
    cfg = lq.config(kda=kda)
    lay = lq.layout(cfg, n)
    offs = [lay.header, lay.counts, lay.full_list, lay.codes, lay.sigma, lay.lambda_, lay.comp_id, lay.comp_line,
            lay.rec_k, lay.rec_u, lay.rec_alpha, lay.total_bytes]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    assert lay.full_list - lay.counts >= 4 * n and lay.codes - lay.full_list >= 4 * n
    assert lay.sigma - lay.codes >= n * 128 * 128
    assert lay.comp_line - lay.comp_id >= 4 * n * lay.comp_id_stride
    assert lay.rec_u - lay.rec_k >= 4 * n * 16 * 128
    assert lay.alpha_stride == (16 * 128 if kda else 16)
    assert lq.state_bytes(cfg, n) == lay.total_bytes
    per_state = (lay.total_bytes - 256) / n
    # GDN: 4 + 4 + 16384 + 512 + 512 + 16 + 2048 + 8192 + 8192 + 64 = 35928 B per head-state, plus padding
    base = 35928 + (8192 - 64 if kda else 0)
    assert base <= per_state <= base + 11 * 256 / n + 1


@pytest.mark.parametrize("field,value,code", [
    ("d_k", 64, lq.ERR_UNSUPPORTED), ("d_v", 256, lq.ERR_UNSUPPORTED), ("window", 0, lq.ERR_UNSUPPORTED),
    ("window", 33, lq.ERR_UNSUPPORTED), ("n_comp", 9, lq.ERR_UNSUPPORTED), ("n_comp", -1, lq.ERR_UNSUPPORTED),
    ("decay_per_key", 2, lq.ERR_INVALID_ARG), ("smooth", 3, lq.ERR_INVALID_ARG),
    ("lambda_floor", 0.0, lq.ERR_INVALID_ARG), ("lambda_floor", float("inf"), lq.ERR_INVALID_ARG),
    ("code_bits", 5, lq.ERR_UNSUPPORTED), ("code_bits", 7, lq.ERR_UNSUPPORTED), ("code_bits", 9, lq.ERR_INVALID_ARG),
    ("code_bits", 0, lq.ERR_INVALID_ARG),
    ("comp_fit", -1, lq.ERR_INVALID_ARG), ("comp_fit", 33, lq.ERR_INVALID_ARG),
    ("comp_block", 1, lq.ERR_INVALID_ARG), ("comp_block", 2, lq.ERR_INVALID_ARG)])
def test_invalid_config_rejected(L, field, value, code):
    cfg = lq.default_config()
    setattr(cfg, field, value)
    assert lq.state_bytes(cfg, 4) == 0
    rc = L.lq_layout(ctypes.byref(cfg), 4, ctypes.byref(lq.Layout()))
    assert rc == code
    assert lq.last_error() != ""


def test_block_fit_needs_fitted_factors_and_changes_the_header_hash(L):
    ok = lq.config(comp_fit=2, comp_block=1)
    assert L.lq_layout(ctypes.byref(ok), 4, ctypes.byref(lq.Layout())) == lq.OK
    assert lq.layout(ok, 4).total_bytes == lq.layout(lq.config(comp_fit=2), 4).total_bytes


def test_invalid_sizes_and_nulls_rejected_on_host(L):
    cfg = lq.default_config()
    assert lq.state_bytes(cfg, -1) == 0
    assert lq.state_bytes(cfg, 2**31) == 0
    assert L.lq_layout(ctypes.byref(cfg), 4, None) == lq.ERR_INVALID_ARG
    assert L.lq_layout(None, 4, ctypes.byref(lq.Layout())) == lq.ERR_INVALID_ARG
    # n_states = 0 is valid and touches no device
    for call in (lambda: L.lq_state_init(ctypes.byref(cfg), None, 0, None, None),
                 lambda: L.lq_fold(ctypes.byref(cfg), None, 0, None),
                 lambda: L.lq_append(ctypes.byref(cfg), None, 0, None, None, None, None, None, None, None),
                 lambda: L.lq_decode_step(ctypes.byref(cfg), None, 0, -1, None, None, None, None, None, None, None),
                 lambda: L.lq_export_state(ctypes.byref(cfg), None, 0, None, None),
                 lambda: L.lq_state_init_range(ctypes.byref(cfg), None, 0, 0, 0, None, None),
                 lambda: L.lq_state_init_range(ctypes.byref(cfg), None, 8, 8, 0, None, None)):
        assert call() == lq.OK
    # a range outside 0..n_states is rejected before the device is looked at
    for first, count in ((-1, 1), (0, -1), (7, 2), (9, 0), (1, 2**40)):
        assert L.lq_state_init_range(ctypes.byref(cfg), None, 8, first, count, None, None) == lq.ERR_INVALID_ARG
        assert "range" in lq.last_error()
    # a bad phase is rejected before anything else is looked at
    assert L.lq_decode_step(ctypes.byref(cfg), None, 0, 16, None, None, None, None, None, None, None) == \
        lq.ERR_INVALID_ARG
    step2 = lambda c, ph: L.lq_decode_step2(ctypes.byref(c), None, 0, ph, *([None] * 10))
    assert step2(cfg, -1) == lq.OK and step2(cfg, 14) == lq.OK
    assert step2(cfg, 15) == lq.ERR_INVALID_ARG  # no room for two records
    one = lq.default_config()
    one.window = 1
    assert step2(one, -1) == lq.ERR_UNSUPPORTED
    rwkv = lambda c, ph: L.lq_decode_step_rwkv7(ctypes.byref(c), None, 0, ph, *([None] * 8))
    kda = lq.config(kda=True)
    assert rwkv(kda, -1) == lq.OK and rwkv(kda, 14) == lq.OK and rwkv(kda, 15) == lq.ERR_INVALID_ARG
    assert rwkv(cfg, -1) == lq.ERR_UNSUPPORTED  # scalar decay


def test_error_message_is_thread_local(L):
    cfg = lq.default_config()
    cfg.window = 99
    L.lq_layout(ctypes.byref(cfg), 1, ctypes.byref(lq.Layout()))
    msg_main = lq.last_error()
    seen = []

    def other():
        seen.append(lq.last_error())

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert "window" in msg_main and seen == [""]


def test_no_gpu_calls_fail_loudly_without_a_device(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = lq.default_config()
    rc = L.lq_fold(ctypes.byref(cfg), ctypes.c_void_p(256), 4, None)
    assert rc in (lq.ERR_CUDA, lq.ERR_INVALID_ARG)
    assert lq.last_error() != ""


def test_debug_wait_hook_rejects_out_of_range_values(L):
    with pytest.raises(lq.LQError):
        lq.debug_set_wait(2_000_000_000, 0, 0)
    with pytest.raises(lq.LQError):
        lq.debug_set_wait(0, -1, 0)
    with pytest.raises(lq.LQError):
        lq.debug_set_wait(0, 0, 4096)
    lq.debug_set_wait(1_000_000, 16, 16)
    lq.debug_set_wait(0, 0, 0)


def test_output_overlapping_the_state_buffer_is_refused(L):
    """o must not overlap the state buffer, which the same kernels read and write; the
    check runs on the host before anything asks the GPU."""
    cfg = lq.config()
    n = 4
    state = 1 << 32
    size = lq.state_bytes(cfg, n)
    far = state + size + (1 << 20)
    q, k, v, a, b = (far + i * 65536 for i in range(5))
    for o in (state + 4096, state + size - 16):
        with pytest.raises(lq.LQError) as e:
            lq.append(cfg, state, n, q, k, v, a, b, o, stream=0)
        assert e.value.code == lq.ERR_INVALID_ARG and "state buffer" in str(e.value)
        with pytest.raises(lq.LQError) as e:
            lq.decode_step(cfg, state, n, q, k, v, a, b, o, phase=0, stream=0)
        assert e.value.code == lq.ERR_INVALID_ARG and "state buffer" in str(e.value)
