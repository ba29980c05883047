"""fo_adamw_step_static, the allocation-free step, for callers that must not
allocate device memory when they step (a loop that reserves all device
memory for its own pools, or code running under an allocator's lock).
Through the C ABI, two consecutive steps must leave exactly the state that
fo_adamw_step leaves on the same inputs.  The list is longer than one launch
of fo_adamw_step (400 tensors), which the static entry point covers in one
launch.  After the first call on the device (its set-up), further calls, in
another kernel variant too, must not change the device memory in use: neither
torch's allocator statistics nor the driver's free memory.

Named to be collected last; it also passes alone in a fresh process.
"""

import ctypes

import pytest
import torch

import quantized_state_optimizer_gb300 as fo
import workloads as W
from quantized_state_optimizer_gb300.optim import FlashAdamWState

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
SLABS = ("param", "rho", "m_codes", "m_scales", "v_codes", "v_scales")


def _state(numels, rho_bits, grad_dtype):
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=grad_dtype, device=DEV)
    for i, n in enumerate(numels):
        if n:
            g = torch.Generator().manual_seed(1000 + i)
            st.init_theta(i, (torch.randn(n, generator=g) * 0.02).to(DEV))
    return st


def _fill_grads(st, numels, t, grad_dtype):
    for i, n in enumerate(numels):
        if n:
            g = torch.Generator().manual_seed(W.grad_seed(7, i, t))
            st.grad_view(i).copy_((torch.randn(n, generator=g) * 1e-3).to(grad_dtype).to(DEV))


@pytest.mark.parametrize("rho_bits,grad_dtype", [(8, torch.bfloat16), (16, torch.float32)])
def test_static_step_equals_fo_adamw_step(rho_bits, grad_dtype):
    numels = [((i * 7919) % 9000) + (i % 5) * 4096 + 1 for i in range(520)]
    numels[3] = 0
    assert len(numels) > fo.fo_max_tensors_per_launch()
    h = W.LLAMA3_8B_HYPER
    a = _state(numels, rho_bits, grad_dtype)
    b = _state(numels, rho_bits, grad_dtype)
    for t in (1, 2):
        _fill_grads(a, numels, t, grad_dtype)
        _fill_grads(b, numels, t, grad_dtype)
        a.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        fo.fo_adamw_step_static(b.fo_tensors(), grad_dtype, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, t,
                                rho_bits)
        torch.cuda.synchronize()
        for k in SLABS:
            x, y = getattr(a, k), getattr(b, k)
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), (k, t)
    assert fo.fo_device_status() == 0


def _memory():
    torch.cuda.synchronize()
    st = torch.cuda.memory_stats()
    return (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0],
            st.get("allocation.all.allocated", 0), st.get("segment.all.allocated", 0))


def test_static_step_allocates_nothing_after_set_up():
    h = W.LLAMA3_8B_HYPER
    numels = [4096 + 17, 7680 * 3, 100]
    a = _state(numels, 8, torch.bfloat16)
    b = _state(numels, 16, torch.float32)  # another kernel variant (grad type, rho width, no decay)
    _fill_grads(a, numels, 1, torch.bfloat16)
    _fill_grads(b, numels, 1, torch.float32)
    arr_a, arr_b = a.fo_tensors(), b.fo_tensors()
    fo.fo_adamw_step_static(arr_a, torch.bfloat16, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 1, 8)
    before = _memory()
    fo.fo_adamw_step_static(arr_a, torch.bfloat16, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 2, 8)
    fo.fo_adamw_step_static(arr_b, torch.float32, h.lr, h.beta1, h.beta2, h.eps, 0.0, 1, 16)
    fo.fo_adamw_step_static(arr_b, torch.float32, h.lr, h.beta1, h.beta2, h.eps, 0.0, 2, 16)
    assert _memory() == before
    assert fo.fo_device_status() == 0


def test_static_step_rejects_too_many_tensors():
    st = _state([64], 8, torch.bfloat16)
    one = st.fo_tensors()[0]
    arr = (fo.FoTensor * (fo.FO_STATIC_MAX_TENSORS + 1))(*([one] * (fo.FO_STATIC_MAX_TENSORS + 1)))
    status = fo.lib().fo_adamw_step_static(arr, len(arr), 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert fo.lib().fo_status_string(status) == b"FO_ERR_TOO_LARGE"
