"""The step kernel certifies results computed with rcp.approx / sqrt.approx /
rsqrt.approx against error bounds that assume at most 2 units in the last
place for each, and a relative error within 4 * 2^-24 of the real result
(the certified codes and the bracket of the 24-bit master's update).
This measures the worst case of each over every positive normal fp32 input on
the device in use and checks it against those assumptions."""

import ctypes
import os
import subprocess

import pytest

from quantized_state_optimizer_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ASSUMED_MAX_ULP = 2
ASSUMED_MAX_REL = 4.0  # units of 2^-24


def test_hardware_approximation_error_within_assumed_bound(tmp_path):
    so = str(tmp_path / "approx_probe.so")
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-Xcompiler", "-fPIC", "-shared", "-o", so,
                    os.path.join(HERE, "native", "approx_probe.cu")], check=True)
    lib = ctypes.CDLL(so)
    out = (ctypes.c_uint * 5)()
    assert lib.approx_probe(out) == 0
    rcp_ulp, sqrt_ulp, rsqrt_u = out[0], out[1], out[2]
    rcp_rel, sqrt_rel = out[3] / 64.0, out[4] / 64.0  # units of 2^-24
    print(f"rcp.approx.ftz max {rcp_ulp} ulp, sqrt.approx.ftz max {sqrt_ulp} ulp, "
          f"rsqrt.approx.ftz max relative error {rsqrt_u} * 2^-24; relative to the real "
          f"result: rcp {rcp_rel:.3f} * 2^-24, sqrt {sqrt_rel:.3f} * 2^-24")
    assert rcp_ulp <= ASSUMED_MAX_ULP and sqrt_ulp <= ASSUMED_MAX_ULP
    # 2 ulp of a result in [2^k, 2^(k+1)) is at most 4 * 2^-24 relative
    assert rsqrt_u <= 2 * ASSUMED_MAX_ULP
    assert 0 < rcp_rel <= ASSUMED_MAX_REL and 0 < sqrt_rel <= ASSUMED_MAX_REL
