"""bench.py's accounting on the CPU: algorithmic bytes per step, the kernel a
format runs in, and the stored DRAM-traffic captures, which must belong to the
kernel sources in the tree (a changed kernel needs a new capture)."""

import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_algorithmic_bytes_of_the_8b_list():
    numels = [s.numel for s in W.llama_tensor_list(W.LLAMA3_8B)]
    assert sum(numels) == 8_030_261_248
    assert bench.algorithmic_bytes(numels) == 98_370_700_288  # 12.25 B per parameter
    # fp32 grad 4 + theta' 2 + 2 + rho 2 + 2 + codes 2 + 2 per element, and the
    # group's two scales read and written
    assert bench.algorithmic_bytes([32], grad_bytes=4, rho_bytes=2) == 32 * 16 + 8


@pytest.mark.parametrize("fmt,optimizer,per_param", [
    ("bf16_rho8:companded", "adamw", 12.25), ("bf16_rho16:linear", "adamw", 14.25),
    ("bf16:f32", "adamw", 22.0), ("f32:f32", "adamw", 26.0),
    ("bf16_rho8:companded", "sgd", 10.125), ("f32:f32", "sgd", 18.0),
])
def test_general_bytes_per_param(fmt, optimizer, per_param):
    assert bench.general_bytes_per_param(*fmt.split(":"), optimizer) == pytest.approx(per_param)


def test_step_kernel_routing():
    assert bench.step_kernel_name(None, "adamw") == "fo::adamw_step_kernel"
    assert bench.step_kernel_name("bf16_rho8:linear", "adamw") == "fo::adamw_step_kernel"
    assert bench.step_kernel_name("bf16_rho8:companded", "adamw") == "fo::adamw_step_kernel"
    assert bench.step_kernel_name("bf16_rho8:f32", "adamw") == "fo::adamw_step_kernel"
    assert bench.step_kernel_name("bf16_rho16:companded", "sgd") == "fo::sgd_step_kernel"
    assert bench.step_kernel_name("bf16:linear", "sgd") == "fo::sgd_step_kernel"
    assert bench.step_kernel_name("f32:companded", "adamw") == "fo::adamw_step_kernel"
    assert bench.step_kernel_name("f32:f32", "sgd") == "fo::sgd_step_kernel"


def test_traffic_capture_is_reported_only_for_the_kernel_sources_it_was_taken_on():
    n = 8_030_261_248
    current = all(
        hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest() == digest
        for rel, digest in bench._CAPTURE_SOURCES.items())
    adamw = bench.captured_traffic(n)
    if not current:
        # the kernel changed since the capture: no traffic figure at all
        assert adamw is None
        return
    # a full launch moves at least the algorithmic bytes less one L2's worth
    assert adamw is not None and 12.25 * n - bench.L2_BYTES <= adamw < 1.01 * 12.25 * n
    assert bench.captured_traffic(n, "fo::adamw_step_kernel", "f32:f32") is None
