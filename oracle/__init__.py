"""CPU oracle of the FlashAdamW step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls it.

The arithmetic lives in ``fo_oracle.c`` (plain C, binary32, no FMA
contraction); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  ctypes releases the GIL during each call, so several
threads may run the oracle on different tensors at once.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fo_oracle.c")
_HDR = os.path.join(_HERE, "fo_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libfo_oracle.so")

# (is_signed, use_sqrt, use_softsign) of the named state specs of the
# quantization page: momentum (Alg. 2), variance (Alg. 3) and the two linear
# ablations.
SPECS = {
    "momentum": (1, 0, 1),
    "variance": (0, 1, 0),
    "momentum_linear": (1, 0, 0),
    "variance_linear": (0, 0, 0),
}

PARAM_BF16_RHO8, PARAM_BF16_RHO16, PARAM_BF16, PARAM_F32 = 0, 1, 2, 3
GRAD_F32, GRAD_BF16 = 0, 1

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libfo_oracle.so`` (gcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest_src:
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L: ctypes.CDLL) -> None:
    p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    for f in (L.fo_oracle_f32_to_f16_array, L.fo_oracle_f16_to_f32_array,
              L.fo_oracle_f32_to_bf16_rne_array):
        f.argtypes = [p, i64, p]
        f.restype = None
    L.fo_oracle_quantize.argtypes = [p, i64, i32, i32, i32, p, p]
    L.fo_oracle_quantize.restype = None
    L.fo_oracle_dequantize.argtypes = [p, p, i64, i32, i32, i32, p]
    L.fo_oracle_dequantize.restype = None
    L.fo_oracle_split.argtypes = [p, i64, i32, p, p]
    L.fo_oracle_split.restype = i32
    L.fo_oracle_reconstruct.argtypes = [p, p, i64, i32, p]
    L.fo_oracle_reconstruct.restype = i32
    L.fo_oracle_adamw_step.argtypes = [i64, p, i32, p, p, i32, p, p, p, p, i32, i32,
                                       d, d, d, d, d, i64]
    L.fo_oracle_adamw_step.restype = i32
    L.fo_oracle_sgd_step.argtypes = [i64, p, i32, p, p, i32, p, p, i32, i32, d, d, d]
    L.fo_oracle_sgd_step.restype = i32


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32).reshape(-1))


def n_groups(n: int) -> int:
    return (n + 31) // 32


# ---------------------------------------------------------------- formats
def f32_to_f16_bits(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty(x.size, dtype=np.uint16)
    lib().fo_oracle_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16).reshape(-1))
    out = np.empty(h.size, dtype=np.float32)
    lib().fo_oracle_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_bf16_rne_bits(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty(x.size, dtype=np.uint16)
    lib().fo_oracle_f32_to_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


# ------------------------------------------------------ quantize/dequantize
def quantize(x, spec: str = "momentum") -> tuple[np.ndarray, np.ndarray]:
    """fp32 -> (codes int8|uint8 [n], fp16 scale bits uint16 [ceil(n/32)])."""
    sg, sq, ss = SPECS[spec]
    x = _f32(x)
    codes = np.empty(x.size, dtype=np.int8 if sg else np.uint8)
    scales = np.empty(n_groups(x.size), dtype=np.uint16)
    lib().fo_oracle_quantize(_ptr(x), x.size, sg, sq, ss, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize(codes, scales, spec: str = "momentum") -> np.ndarray:
    sg, sq, ss = SPECS[spec]
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.int8 if sg else np.uint8).reshape(-1))
    scales = np.ascontiguousarray(np.asarray(scales, dtype=np.uint16).reshape(-1))
    assert scales.size >= n_groups(codes.size)
    out = np.empty(codes.size, dtype=np.float32)
    lib().fo_oracle_dequantize(_ptr(codes), _ptr(scales), codes.size, sg, sq, ss, _ptr(out))
    return out


# ---------------------------------------------------------- split / recon
def rho_dtype(master_bits: int):
    if master_bits not in (24, 32):
        raise ValueError(f"bad master_bits {master_bits} (24 or 32)")
    return {24: np.int8, 32: np.int16}[master_bits]


def split(theta, master_bits: int = 24) -> tuple[np.ndarray, np.ndarray]:
    """fp32 -> (bf16 bits uint16 [n], rho int8|int16 [n])."""
    x = _f32(theta)
    hi = np.empty(x.size, dtype=np.uint16)
    rho = np.empty(x.size, dtype=rho_dtype(master_bits))
    rc = lib().fo_oracle_split(_ptr(x), x.size, master_bits, _ptr(hi), _ptr(rho))
    if rc != 0:
        raise ValueError(f"bad master_bits {master_bits}")
    return hi, rho


def reconstruct(theta_bf16, rho, master_bits: int = 24) -> np.ndarray:
    hi = np.ascontiguousarray(np.asarray(theta_bf16, dtype=np.uint16).reshape(-1))
    rho = np.ascontiguousarray(np.asarray(rho, dtype=rho_dtype(master_bits)).reshape(-1))
    assert hi.size == rho.size
    out = np.empty(hi.size, dtype=np.float32)
    rc = lib().fo_oracle_reconstruct(_ptr(hi), _ptr(rho), hi.size, master_bits, _ptr(out))
    if rc != 0:
        raise ValueError(f"bad master_bits {master_bits}")
    return out


# ------------------------------------------------------------- the step
class TensorState:
    """One parameter's optimizer state as plain numpy arrays (flat).

    ``param`` holds bf16 bits (uint16) or fp32; ``rho`` int8/int16 or None;
    ``m``/``v`` are codes (int8/uint8) with fp16 scale bits, or fp32 arrays
    when states are not quantized.
    """

    def __init__(self, param, rho, m, m_scales, v, v_scales, param_kind: int):
        self.param, self.rho = param, rho
        self.m, self.m_scales, self.v, self.v_scales = m, m_scales, v, v_scales
        self.param_kind = param_kind

    @property
    def numel(self) -> int:
        return self.param.size

    @classmethod
    def init(cls, theta, master_bits: int | None = 24, quantize_states: bool = True,
             param_dtype: str = "bf16") -> "TensorState":
        """Initial state: states are zeros (quantized zeros are all-zero codes and
        scales) and theta is split into (theta', rho) (Alg. 4 initialisation)."""
        theta = _f32(theta)
        n = theta.size
        if quantize_states:
            m, ms = quantize(np.zeros(n, np.float32), "momentum")
            v, vs = quantize(np.zeros(n, np.float32), "variance")
        else:
            m, ms = np.zeros(n, np.float32), np.zeros(0, np.uint16)
            v, vs = np.zeros(n, np.float32), np.zeros(0, np.uint16)
        if param_dtype == "f32":
            return cls(theta.copy(), None, m, ms, v, vs, PARAM_F32)
        if master_bits is None:
            return cls(f32_to_bf16_rne_bits(theta), None, m, ms, v, vs, PARAM_BF16)
        hi, rho = split(theta, master_bits)
        kind = PARAM_BF16_RHO8 if master_bits == 24 else PARAM_BF16_RHO16
        return cls(hi, rho, m, ms, v, vs, kind)

    def copy(self) -> "TensorState":
        c = lambda a: None if a is None else a.copy()  # noqa: E731
        return TensorState(c(self.param), c(self.rho), c(self.m), c(self.m_scales), c(self.v),
                           c(self.v_scales), self.param_kind)

    def theta(self) -> np.ndarray:
        """The fp32 master weight this state represents."""
        if self.param_kind == PARAM_F32:
            return self.param.copy()
        if self.param_kind == PARAM_BF16:
            return (self.param.astype(np.uint32) << 16).view(np.float32)
        return reconstruct(self.param, self.rho, 24 if self.param_kind == PARAM_BF16_RHO8 else 32)


def adamw_step(st: TensorState, grad, step: int, lr: float, beta1: float, beta2: float,
               eps: float, weight_decay: float, quantize_states: bool = True,
               companded: bool = True) -> None:
    """One FlashAdamW step of one tensor, in place.  ``grad`` is fp32 or bf16
    bits (uint16)."""
    grad = np.ascontiguousarray(np.asarray(grad).reshape(-1))
    if grad.dtype == np.float32:
        gk = GRAD_F32
    elif grad.dtype == np.uint16:
        gk = GRAD_BF16
    else:
        raise TypeError(f"grad dtype {grad.dtype}")
    assert grad.size == st.numel
    null = 0
    rc = lib().fo_oracle_adamw_step(
        st.numel, _ptr(st.param), st.param_kind, _ptr(st.rho) if st.rho is not None else null,
        _ptr(grad), gk, _ptr(st.m), _ptr(st.m_scales) if st.m_scales.size else null,
        _ptr(st.v), _ptr(st.v_scales) if st.v_scales.size else null,
        int(quantize_states), int(companded), lr, beta1, beta2, eps, weight_decay, step)
    if rc != 0:
        raise RuntimeError("oracle adamw_step failed")


def sgd_step(st: TensorState, grad, lr: float, momentum: float, weight_decay: float,
             quantize_states: bool = True, companded: bool = True) -> None:
    """One FlashSGD step of one tensor, in place (the momentum buffer lives in
    ``st.m`` / ``st.m_scales``; ``st.v`` is unused).  ``grad`` is fp32 or bf16
    bits (uint16).  The update is the reading stated in fo_oracle.h [B]."""
    grad = np.ascontiguousarray(np.asarray(grad).reshape(-1))
    if grad.dtype == np.float32:
        gk = GRAD_F32
    elif grad.dtype == np.uint16:
        gk = GRAD_BF16
    else:
        raise TypeError(f"grad dtype {grad.dtype}")
    assert grad.size == st.numel
    rc = lib().fo_oracle_sgd_step(
        st.numel, _ptr(st.param), st.param_kind, _ptr(st.rho) if st.rho is not None else 0,
        _ptr(grad), gk, _ptr(st.m), _ptr(st.m_scales) if st.m_scales.size else 0,
        int(quantize_states), int(companded), lr, momentum, weight_decay)
    if rc != 0:
        raise RuntimeError("oracle sgd_step failed")


# ------------------------------------------------------------ statistics
def nmse(orig, recon) -> float:
    """Normalised MSE in binary64 (quantization page, ``nmse``; 0 for a zero signal)."""
    o = np.asarray(orig, dtype=np.float64).reshape(-1)
    r = np.asarray(recon, dtype=np.float64).reshape(-1)
    denom = float(np.mean(o * o))
    if denom == 0.0:
        return 0.0
    return float(np.mean((o - r) ** 2)) / denom
