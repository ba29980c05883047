"""The C ABI library builds, loads without a GPU, exports every symbol that
include/fo.h declares, and rejects bad arguments on the host before any CUDA
call (no kernel runs here)."""

import ctypes
import os
import re

import pytest

import quantized_state_optimizer_gb300 as fo
from quantized_state_optimizer_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fo.h")

OK, INVALID, MISALIGNED, CUDA, ALIAS = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    B.build()
    return fo.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fo_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("fo_quantize", "fo_dequantize", "fo_split", "fo_reconstruct", "fo_adamw_step"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    assert L.fo_status_string(0) == b"FO_OK"
    assert L.fo_status_string(4) == b"FO_ERR_ALIAS"
    assert L.fo_last_cuda_error() == b""
    assert L.fo_max_tensors_per_launch() >= 291


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def test_pair_argument_errors(L):
    assert L.fo_quantize(FAKE, -1, 0, FAKE, FAKE, None) == INVALID
    assert L.fo_quantize(FAKE, 10, 7, FAKE, FAKE, None) == INVALID
    assert L.fo_quantize(None, 10, 0, FAKE, FAKE, None) == INVALID
    assert L.fo_quantize(FAKE + 4, 10, 0, FAKE, FAKE, None) == MISALIGNED
    assert L.fo_quantize(FAKE, 10, 0, FAKE, FAKE + 2, None) == MISALIGNED
    assert L.fo_quantize(None, 0, 0, None, None, None) == OK  # empty: no-op
    assert L.fo_dequantize(FAKE, FAKE, 10, 9, FAKE, None) == INVALID
    assert L.fo_dequantize(FAKE, FAKE, 10, 0, FAKE + 8, None) == MISALIGNED
    assert L.fo_split(FAKE, 10, 12, FAKE, FAKE, None) == INVALID
    assert L.fo_split(FAKE, 10, 8, FAKE, FAKE + 1, None) == MISALIGNED
    assert L.fo_reconstruct(FAKE, FAKE, 10, 8, None, None) == INVALID
    assert L.fo_reconstruct(FAKE, FAKE, 0, 16, None, None) == OK


def test_wait_timeout_probe_rejects_bad_poll_counts(L):
    assert L.fo_check_wait_timeout(0, None) == INVALID
    assert L.fo_check_wait_timeout((1 << 22) + 1, None) == INVALID


def _t(base, n, grad=None, stride=1 << 20):
    return fo.FoTensor(base, base + stride, grad if grad is not None else base + 2 * stride,
                       base + 3 * stride, base + 4 * stride, base + 5 * stride, base + 6 * stride, n)


def _step(L, ts, **kw):
    arr = (fo.FoTensor * max(len(ts), 1))(*ts)
    a = dict(grad_dtype=1, lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, step=1, rho=8)
    a.update(kw)
    return L.fo_adamw_step(arr, len(ts), a["grad_dtype"], a["lr"], a["b1"], a["b2"], a["eps"],
                           a["wd"], a["step"], a["rho"], None)


def test_step_argument_errors(L):
    t = _t(1 << 32, 1000)
    assert _step(L, [t], step=0) == INVALID
    assert _step(L, [t], rho=12) == INVALID
    assert _step(L, [t], grad_dtype=5) == INVALID
    assert _step(L, [t], b1=1.0) == INVALID
    assert _step(L, [t], b2=-0.1) == INVALID
    assert _step(L, [t], lr=float("nan")) == INVALID
    assert _step(L, [t], eps=float("inf")) == INVALID
    assert _step(L, [_t(1 << 32, -5)]) == INVALID
    bad = _t(1 << 32, 1000)
    bad.m_codes = 0
    assert _step(L, [bad]) == INVALID
    mis = _t(1 << 32, 1000)
    mis.v_scales += 2
    assert _step(L, [mis]) == MISALIGNED
    assert L.fo_adamw_step(None, 3, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == INVALID
    # an empty list, or only empty tensors, is a no-op
    assert L.fo_adamw_step(None, 0, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == OK
    assert _step(L, [_t(0, 0)]) == OK


def test_step_alias_detection(L):
    base = 1 << 32
    # two tensors whose param buffers overlap
    a = _t(base, 1000)
    b = _t(base + (1 << 24), 1000)
    b.param = a.param + 512
    assert _step(L, [a, b]) == ALIAS
    # a written buffer overlapping a grad
    c = _t(base, 1000)
    c.grad = c.rho + 16
    assert _step(L, [c]) == ALIAS
    # scales too short to hold ceil(n/32) entries overlap the next buffer
    d = _t(base, 1000, stride=32)
    assert _step(L, [d]) == ALIAS


def test_static_step_host_checks(L):
    """fo_adamw_step_static: the size limit comes first, then the same argument
    and alias checks as fo_adamw_step, all before any CUDA call."""
    big = (fo.FoTensor * (fo.FO_STATIC_MAX_TENSORS + 1))()
    assert L.fo_adamw_step_static(big, len(big), 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == 5
    assert L.fo_status_string(5) == b"FO_ERR_TOO_LARGE"
    t = _t(1 << 32, 1000)
    arr = (fo.FoTensor * 1)(t)
    assert L.fo_adamw_step_static(arr, 1, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 0, 8, None) == INVALID
    mis = _t(1 << 32, 1000)
    mis.v_scales += 2
    assert L.fo_adamw_step_static((fo.FoTensor * 1)(mis), 1, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == MISALIGNED
    a = _t(1 << 32, 1000)
    b = _t((1 << 32) + (1 << 24), 1000)
    b.param = a.param + 512
    assert L.fo_adamw_step_static((fo.FoTensor * 2)(a, b), 2, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == ALIAS
    assert L.fo_adamw_step_static(None, 0, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8, None) == OK


def test_general_step_host_checks(L):
    """fo_adamw_step_general rejects bad formats and arguments before any CUDA call."""
    t = fo.FoTensorGeneral(1 << 32, 0, (1 << 32) + (2 << 20), (1 << 32) + (3 << 20), 0,
                           (1 << 32) + (5 << 20), 0, 1000)
    arr = (fo.FoTensorGeneral * 1)(t)
    call = lambda pf, sf, **kw: L.fo_adamw_step_general(  # noqa: E731
        arr, 1, pf, sf, kw.get("gd", 1), 1e-3, 0.9, 0.999, 1e-8, 0.0, kw.get("step", 1), None)
    assert call(4, 0) == INVALID          # no such parameter format
    assert call(0, 3) == INVALID          # no such state format
    assert call(3, 2, gd=7) == INVALID    # no such grad dtype
    assert call(3, 2, step=0) == INVALID
    assert call(0, 2) == INVALID          # a split needs rho
    assert call(3, 0) == INVALID          # quantized states need scales
    assert L.fo_adamw_step_general(None, 0, 3, 2, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None) == OK


def test_sgd_step_host_checks(L):
    """fo_sgd_step needs no v buffers, and rejects bad arguments before any CUDA call."""
    t = fo.FoTensorGeneral(1 << 32, 0, (1 << 32) + (2 << 20), (1 << 32) + (3 << 20), 0, 0, 0, 1000)
    arr = (fo.FoTensorGeneral * 1)(t)
    assert L.fo_sgd_step(arr, 1, 3, 0, 1, 1e-2, 0.9, 0.0, None) == INVALID   # quantized buffer needs scales
    assert L.fo_sgd_step(arr, 1, 4, 2, 1, 1e-2, 0.9, 0.0, None) == INVALID   # no such parameter format
    assert L.fo_sgd_step(arr, 1, 3, 2, 1, float("nan"), 0.9, 0.0, None) == INVALID
    assert L.fo_sgd_step(None, 0, 3, 2, 1, 1e-2, 0.9, 0.0, None) == OK
