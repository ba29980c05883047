"""The fused step's correctly rounded division and square root (fo_device.cuh:
div_const2, sqrt_cert2, div_cert2 in their packed f32x2 form: a hardware
approximation, FMA residuals and one rounding, after Markstein) against the
device's IEEE division and square root, bit for bit:

- the square root over every input of its domain (+0 and [2^-95, 2^100]);
- division by a launch constant over every dividend of its domain, for the
  bias corrections of the workloads' betas at many steps, divisors with an
  all-ones significand, powers of two and random divisors in [2^-20, 1];
- general division over every numerator significand of one binade, both
  signs, for 1024 divisors in [2^-36, 2^21] (random significands, all-ones
  significands, powers of two, the typical sqrt(v_hat) + eps values).

A result whose certificate fails is not compared (the step then recomputes
its thread through the IEEE chain); the rate of failed certificates is
checked to be small, so that the exact fallback stays rare."""

import ctypes
import os
import subprocess

import numpy as np
import pytest

from quantized_state_optimizer_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("exact") / "exact_probe.so")
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
                    "-I", B.CSRC, "-I", B.INCLUDE, "-o", so, os.path.join(HERE, "native", "exact_probe.cu")],
                   check=True)
    return ctypes.CDLL(so)


def f32(xs):
    return np.ascontiguousarray(np.asarray(xs, dtype=np.float32))


def test_sqrt_every_input(probe):
    out = (ctypes.c_ulonglong * 3)()
    assert probe.probe_sqrt(out) == 0
    checked, bad, unsure = out[0], out[1], out[2]
    print(f"sqrt: {checked} inputs, {bad} mismatches, {unsure} uncertain")
    assert checked == 0x71800000 - 0x10000000 + 2
    assert bad == 0
    assert unsure < 1e-5 * checked


def bias_corrections():
    out = []
    for beta in (0.9, 0.95, 0.99, 0.999, 0.9999):
        for t in list(range(1, 40)) + [50, 100, 200, 500, 1000, 5000, 20000]:
            bc = np.float32(1.0 - beta ** t)
            if 2.0 ** -20 <= bc <= 1.0:
                out.append(bc)
    return out


def test_division_by_launch_constants(probe):
    rng = np.random.default_rng(5)
    divs = bias_corrections()
    divs += [np.float32(1.0), np.float32(0.5), np.float32(2.0 ** -20), np.float32(2.0 ** -7)]
    # all-ones significands (the hardest case for a reciprocal)
    divs += [np.float32(np.ldexp(2.0 - 2.0 ** -23, -e)) for e in (1, 3, 9, 20)]
    divs += list(np.ldexp(rng.uniform(1.0, 2.0, 24), -rng.integers(1, 21, 24)).astype(np.float32))
    divs = f32(sorted(set(float(d) for d in divs)))
    assert np.all((divs >= 2.0 ** -20) & (divs <= 1.0))
    out = (ctypes.c_ulonglong * (3 * len(divs)))()
    assert probe.probe_div_const(divs.ctypes.data_as(ctypes.c_void_p), len(divs), out) == 0
    res = np.array(out[:], dtype=np.uint64).reshape(-1, 3)
    bad = {float(d): int(r[1]) for d, r in zip(divs, res) if r[1]}
    print(f"division by {len(divs)} constants, {int(res[:, 0].sum())} quotients")
    assert not bad, f"mismatches per divisor: {bad}"


def test_general_division(probe):
    rng = np.random.default_rng(6)
    n = 1024
    sig = rng.uniform(1.0, 2.0, n)
    sig[:64] = 2.0 - 2.0 ** -23  # all-ones significands
    sig[64:96] = 1.0  # powers of two
    exps = rng.integers(-36, 21, n)
    divs = np.ldexp(sig, exps)
    # sqrt(v_hat) + eps of the workloads: sqrt of 1e-7 .. 1e-5 plus 1e-8
    divs[96:256] = np.sqrt(rng.uniform(1e-8, 1e-5, 160)) + 1e-8
    divs = f32(np.clip(divs, 2.0 ** -36, 2.0 ** 21))
    out = (ctypes.c_ulonglong * 3)()
    assert probe.probe_div_cert(divs.ctypes.data_as(ctypes.c_void_p), n, out) == 0
    checked, bad, unsure = out[0], out[1], out[2]
    print(f"general division: {checked} quotients, {bad} mismatches, {unsure} uncertain")
    assert checked == n << 24
    assert bad == 0
    assert unsure < 1e-5 * checked
