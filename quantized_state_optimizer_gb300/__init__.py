"""GB300-native FlashAdamW: quantized optimizer states and split master weights.

Thin Python binding of ``libfo.so`` (C ABI declared in ``include/fo.h``).
Each function here has the name of a C entry point and only marshals
arguments -- torch tensors to device pointers, the current CUDA stream to a
``cudaStream_t`` -- before calling it; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: if the library has not
been built, importing this package succeeds but every call raises.

Build with ``python -m quantized_state_optimizer_gb300.build`` (or
``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as _LIB_PATH

__all__ = [
    "FoError", "SPECS", "fo_quantize", "fo_dequantize", "fo_split", "fo_reconstruct",
    "fo_adamw_step", "fo_adamw_step_static", "FO_STATIC_MAX_TENSORS", "fo_adamw_step_general",
    "FoTensorGeneral", "PARAM_FORMATS", "STATE_FORMATS", "fo_sgd_step", "fo_max_tensors_per_launch",
    "fo_device_status", "fo_check_wait_timeout", "FoTensor", "lib", "lib_path",
]

SPECS = {"momentum": 0, "variance": 1, "momentum_linear": 2, "variance_linear": 3}
_SIGNED = {0: True, 1: False, 2: True, 3: False}
FO_DT_F32, FO_DT_BF16 = 0, 1
FO_STATIC_MAX_TENSORS = 1024  # include/fo.h
# fo_param_format / fo_state_format of include/fo.h
PARAM_FORMATS = {"bf16_rho8": 0, "bf16_rho16": 1, "bf16": 2, "f32": 3}
STATE_FORMATS = {"companded": 0, "linear": 1, "f32": 2}


class FoError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        name = _lib.fo_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


class FoTensor(ctypes.Structure):
    """``fo_tensor`` of include/fo.h: one parameter tensor's device buffers."""
    _fields_ = [
        ("param", ctypes.c_void_p),
        ("rho", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("m_codes", ctypes.c_void_p),
        ("m_scales", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
    ]


class FoTensorGeneral(ctypes.Structure):
    """``fo_tensor_general`` of include/fo.h: one tensor's buffers in any format."""
    _fields_ = [
        ("param", ctypes.c_void_p),
        ("rho", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("m", ctypes.c_void_p),
        ("m_scales", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
    ]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libfo.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -m quantized_state_optimizer_gb300.build)")
        L = ctypes.CDLL(_LIB_PATH)
        p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.fo_status_string.argtypes = [i32]
        L.fo_status_string.restype = ctypes.c_char_p
        L.fo_last_cuda_error.argtypes = []
        L.fo_last_cuda_error.restype = ctypes.c_char_p
        L.fo_quantize.argtypes = [p, i64, i32, p, p, p]
        L.fo_dequantize.argtypes = [p, p, i64, i32, p, p]
        L.fo_split.argtypes = [p, i64, i32, p, p, p]
        L.fo_reconstruct.argtypes = [p, p, i64, i32, p, p]
        L.fo_adamw_step.argtypes = [ctypes.POINTER(FoTensor), i32, i32, d, d, d, d, d, i64, i32, p]
        L.fo_adamw_step_static.argtypes = [ctypes.POINTER(FoTensor), i32, i32, d, d, d, d, d, i64, i32, p]
        L.fo_adamw_step_general.argtypes = [ctypes.POINTER(FoTensorGeneral), i32, i32, i32, i32, d, d, d, d, d,
                                            i64, p]
        L.fo_sgd_step.argtypes = [ctypes.POINTER(FoTensorGeneral), i32, i32, i32, i32, d, d, d, p]
        L.fo_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.fo_device_status.restype = i32
        L.fo_check_wait_timeout.argtypes = [ctypes.c_uint32, p]
        L.fo_check_wait_timeout.restype = i32
        L.fo_max_tensors_per_launch.argtypes = []
        L.fo_max_tensors_per_launch.restype = i32
        for f in ("fo_quantize", "fo_dequantize", "fo_split", "fo_reconstruct", "fo_adamw_step",
                  "fo_adamw_step_static", "fo_adamw_step_general", "fo_sgd_step"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, status: int) -> None:
    if status != 0:
        detail = lib().fo_last_cuda_error().decode() if status == 3 else ""
        raise FoError(fn, status, detail)


def _dev(t: torch.Tensor, name: str, dtype=None, numel: int | None = None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, need {numel}")
    return t.data_ptr()


def n_groups(n: int) -> int:
    return (n + 31) // 32


def _spec(spec) -> int:
    return SPECS[spec] if isinstance(spec, str) else int(spec)


# ----------------------------------------------------------------- pairs
def fo_quantize(x: torch.Tensor, spec, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """Group-32 quantize fp32 ``x`` into ``codes`` (int8 / uint8) and fp16 ``scales``."""
    s = _spec(spec)
    n = x.numel()
    cdt = torch.int8 if _SIGNED.get(s, True) else torch.uint8
    _check("fo_quantize", lib().fo_quantize(
        _dev(x, "x", torch.float32), n, s, _dev(codes, "codes", cdt, n),
        _dev(scales, "scales", (torch.float16, torch.int16, torch.uint16), n_groups(n)), _stream(stream)))


def fo_dequantize(codes: torch.Tensor, scales: torch.Tensor, spec, out: torch.Tensor, stream=None) -> None:
    s = _spec(spec)
    n = codes.numel()
    cdt = torch.int8 if _SIGNED.get(s, True) else torch.uint8
    _check("fo_dequantize", lib().fo_dequantize(
        _dev(codes, "codes", cdt), _dev(scales, "scales", (torch.float16, torch.int16, torch.uint16), n_groups(n)),
        n, s, _dev(out, "out", torch.float32, n), _stream(stream)))


def _rho_dtype(rho_bits: int):
    return {8: torch.int8, 16: torch.int16}.get(rho_bits)


def fo_split(theta: torch.Tensor, rho_bits: int, theta_bf16: torch.Tensor, rho: torch.Tensor,
             stream=None) -> None:
    n = theta.numel()
    _check("fo_split", lib().fo_split(
        _dev(theta, "theta", torch.float32), n, rho_bits,
        _dev(theta_bf16, "theta_bf16", (torch.bfloat16, torch.int16, torch.uint16), n),
        _dev(rho, "rho", _rho_dtype(rho_bits) or rho.dtype, n), _stream(stream)))


def fo_reconstruct(theta_bf16: torch.Tensor, rho: torch.Tensor, rho_bits: int, theta: torch.Tensor,
                   stream=None) -> None:
    n = theta_bf16.numel()
    _check("fo_reconstruct", lib().fo_reconstruct(
        _dev(theta_bf16, "theta_bf16", (torch.bfloat16, torch.int16, torch.uint16)),
        _dev(rho, "rho", _rho_dtype(rho_bits) or rho.dtype, n), n, rho_bits,
        _dev(theta, "theta", torch.float32, n), _stream(stream)))


# ------------------------------------------------------------------ step
def fo_max_tensors_per_launch() -> int:
    return lib().fo_max_tensors_per_launch()


def fo_check_wait_timeout(polls: int = 4096, stream=None) -> None:
    """One block whose bounded wait on a barrier that nothing completes runs out
    after ``polls`` polls and sets the timeout bit that ``fo_device_status``
    reports (failure detection, exercised without a fault)."""
    _check("fo_check_wait_timeout", lib().fo_check_wait_timeout(ctypes.c_uint32(int(polls)), _stream(stream)))


def fo_device_status() -> int:
    """Device status word of the step kernel (0 = no bounded wait ran out); clears it.
    Synchronizes with the device."""
    out = ctypes.c_uint32(0)
    _check("fo_device_status", lib().fo_device_status(ctypes.byref(out)))
    return out.value


def make_fo_tensor(param: torch.Tensor, rho: torch.Tensor, grad: torch.Tensor, m_codes: torch.Tensor,
                   m_scales: torch.Tensor, v_codes: torch.Tensor, v_scales: torch.Tensor) -> FoTensor:
    """Marshal one parameter's buffers (all flat views of CUDA tensors)."""
    n = param.numel()
    g = n_groups(n)
    return FoTensor(
        _dev(param, "param", (torch.bfloat16, torch.int16, torch.uint16)),
        _dev(rho, "rho", (torch.int8, torch.int16), n),
        _dev(grad, "grad", (torch.float32, torch.bfloat16), n),
        _dev(m_codes, "m_codes", torch.int8, n),
        _dev(m_scales, "m_scales", (torch.float16, torch.int16, torch.uint16), g),
        _dev(v_codes, "v_codes", torch.uint8, n),
        _dev(v_scales, "v_scales", (torch.float16, torch.int16, torch.uint16), g),
        n)


def _step_args(tensors, grad_dtype):
    if isinstance(grad_dtype, torch.dtype):
        grad_dtype = FO_DT_BF16 if grad_dtype == torch.bfloat16 else FO_DT_F32
    if isinstance(tensors, ctypes.Array):
        return tensors, len(tensors), int(grad_dtype)
    tensors = list(tensors)
    return (FoTensor * max(len(tensors), 1))(*tensors), len(tensors), int(grad_dtype)


def fo_adamw_step(tensors, grad_dtype, lr: float, beta1: float, beta2: float, eps: float,
                  weight_decay: float, step: int, rho_bits: int, stream=None) -> None:
    """One fused FlashAdamW step over a list of ``FoTensor`` (or a ctypes array of them)."""
    arr, count, gdt = _step_args(tensors, grad_dtype)
    _check("fo_adamw_step", lib().fo_adamw_step(
        arr, count, gdt, float(lr), float(beta1), float(beta2), float(eps),
        float(weight_decay), int(step), int(rho_bits), _stream(stream)))


def fo_adamw_step_static(tensors, grad_dtype, lr: float, beta1: float, beta2: float, eps: float,
                         weight_decay: float, step: int, rho_bits: int, stream=None) -> None:
    """``fo_adamw_step`` for at most ``FO_STATIC_MAX_TENSORS`` tensors in one
    launch, with the list in the library's fixed device array: the call
    allocates nothing (see include/fo.h for its set-up and sharing rules)."""
    arr, count, gdt = _step_args(tensors, grad_dtype)
    _check("fo_adamw_step_static", lib().fo_adamw_step_static(
        arr, count, gdt, float(lr), float(beta1), float(beta2), float(eps),
        float(weight_decay), int(step), int(rho_bits), _stream(stream)))


def fo_adamw_step_general(tensors, param_format, state_format, grad_dtype, lr: float, beta1: float,
                          beta2: float, eps: float, weight_decay: float, step: int, stream=None) -> None:
    """The step in any parameter / state format (``PARAM_FORMATS``, ``STATE_FORMATS``)
    over a list of ``FoTensorGeneral`` (or a ctypes array of them)."""
    if isinstance(grad_dtype, torch.dtype):
        grad_dtype = FO_DT_BF16 if grad_dtype == torch.bfloat16 else FO_DT_F32
    pf = PARAM_FORMATS[param_format] if isinstance(param_format, str) else int(param_format)
    sf = STATE_FORMATS[state_format] if isinstance(state_format, str) else int(state_format)
    if isinstance(tensors, ctypes.Array):
        arr, count = tensors, len(tensors)
    else:
        tensors = list(tensors)
        count = len(tensors)
        arr = (FoTensorGeneral * max(count, 1))(*tensors)
    _check("fo_adamw_step_general", lib().fo_adamw_step_general(
        arr, count, pf, sf, int(grad_dtype), float(lr), float(beta1), float(beta2), float(eps),
        float(weight_decay), int(step), _stream(stream)))


def fo_sgd_step(tensors, param_format, state_format, grad_dtype, lr: float, momentum: float,
                weight_decay: float, stream=None) -> None:
    """One FlashSGD step over a list of ``FoTensorGeneral`` (the momentum buffer
    in ``m`` / ``m_scales``; see include/fo.h for the update)."""
    if isinstance(grad_dtype, torch.dtype):
        grad_dtype = FO_DT_BF16 if grad_dtype == torch.bfloat16 else FO_DT_F32
    pf = PARAM_FORMATS[param_format] if isinstance(param_format, str) else int(param_format)
    sf = STATE_FORMATS[state_format] if isinstance(state_format, str) else int(state_format)
    if isinstance(tensors, ctypes.Array):
        arr, count = tensors, len(tensors)
    else:
        tensors = list(tensors)
        count = len(tensors)
        arr = (FoTensorGeneral * max(count, 1))(*tensors)
    _check("fo_sgd_step", lib().fo_sgd_step(
        arr, count, pf, sf, int(grad_dtype), float(lr), float(momentum), float(weight_decay), _stream(stream)))
