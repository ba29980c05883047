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


@pytest.mark.parametrize("per_tensor", [False, True])
def test_bench_steps_cycle_the_gradient_sets(per_tensor):
    """Step t of the timed loop launches over gradient set (t - 1) mod 2: every
    tensor's grad pointer lies in that set's slab at the tensor's own offset,
    and the other state pointers are the same in both sets.  Host memory only;
    nothing is launched."""
    import torch
    from quantized_state_optimizer_gb300.optim import FlashAdamWState
    numels = [100, 3000, (1 << 20) + 5, 4096, 7]
    st = FlashAdamWState(numels, rho_bits=8, device="cpu")
    slabs = [st.grad, torch.zeros_like(st.grad)]
    steps = bench.BenchSteps(st, slabs, per_tensor=per_tensor)
    full = st.fo_tensors()
    big = [i for i, n in enumerate(numels) if n >= 1 << 20]
    small = [i for i, n in enumerate(numels) if n < 1 << 20]
    order = (big + small) if per_tensor else list(range(len(numels)))
    assert steps.launches_per_step == (len(big) + 1 if per_tensor else 1)
    for t in (1, 2, 3, 4):
        k = (t - 1) % 2
        launched = [ft for arr in steps.sets[k] for ft in arr]
        assert len(launched) == len(numels)
        for ft, i in zip(launched, order):
            off = st.grad_view(i).storage_offset() * st.grad.element_size()
            assert ft.grad == slabs[k].data_ptr() + off
            assert (ft.param, ft.rho, ft.m_codes, ft.v_codes, ft.numel) == \
                (full[i].param, full[i].rho, full[i].m_codes, full[i].v_codes, full[i].numel)


def test_general_state_gradient_sets():
    """The ablation-format state builds its argument array for any grad slab."""
    import torch
    st = bench.GeneralState([33, 4096, 5], "f32", "linear", "cpu")
    other = torch.zeros_like(st.grad)
    arr = st.grad_array(other)
    for i, n in enumerate(st.numels):
        assert arr[i].grad == other.data_ptr() + st.offs[i] * 2
        assert arr[i].param == st.arr[i].param and arr[i].numel == n
