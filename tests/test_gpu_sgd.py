"""FlashSGD (fo_sgd_step) against the oracle's FlashSGD step, bit for bit, in
every parameter and state format, and the FlashSGD optimizer on a small
model."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_state_optimizer_gb300 as fo
import workloads as W
from quantized_state_optimizer_gb300 import FoTensorGeneral
from quantized_state_optimizer_gb300.optim import FlashSGD
from test_gpu_general import DevTensor, _oracle_state, _same, _theta

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
NUMELS = [1, 33, 4096 + 17, 12345, 0, 64]


def _grad(i, t, n, dtype):
    g = torch.Generator().manual_seed(W.grad_seed(66, i, t))
    x = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g)) * 1e-3
    return x if dtype == torch.float32 else x.to(torch.bfloat16)


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sf", ["companded", "linear", "f32"])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16", "bf16", "f32"])
def test_sgd_step_matches_oracle(pf, sf, grad_dtype):
    lr, mu, wd = 1e-2, 0.9, 0.01
    thetas = [_theta(i, n) for i, n in enumerate(NUMELS)]
    dev = [DevTensor(t, pf, sf, grad_dtype) for t in thetas]
    refs = [_oracle_state(t, pf, sf) for t in thetas]
    arr = (FoTensorGeneral * len(dev))(*[d.ft() for d in dev])
    for k in range(len(arr)):  # one state: v is not used
        arr[k].v = None
        arr[k].v_scales = None
    for t in range(1, 4):
        for i, n in enumerate(NUMELS):
            if n == 0:
                continue
            g = _grad(i, t, n, grad_dtype)
            dev[i].grad.copy_(g.to(DEV))
            gn = g.numpy() if grad_dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16)
            O.sgd_step(refs[i], gn, lr, mu, wd, quantize_states=sf != "f32", companded=sf == "companded")
        fo.fo_sgd_step(arr, pf, sf, grad_dtype, lr, mu, wd)
        torch.cuda.synchronize()
        for i, n in enumerate(NUMELS):
            if n == 0:
                continue
            got, r = dev[i].host(), refs[i]
            ctx = (pf, sf, str(grad_dtype), i, t)
            _same(got["param"], r.param, ctx + ("param",))
            if r.rho is not None:
                _same(got["rho"], r.rho, ctx + ("rho",))
            _same(got["m"], r.m, ctx + ("m",))
            if sf != "f32":
                _same(got["ms"], r.m_scales, ctx + ("m_scales",))


def test_flash_sgd_optimizer_matches_oracle():
    torch.manual_seed(0)
    net = torch.nn.Sequential(torch.nn.Linear(48, 80), torch.nn.Tanh(), torch.nn.Linear(80, 16)).to(
        device=DEV, dtype=torch.bfloat16)
    params = list(net.parameters())
    refs = [O.TensorState.init(p.detach().float().cpu().reshape(-1).numpy(), master_bits=24) for p in params]
    opt = FlashSGD(net.parameters(), lr=5e-2, momentum=0.9, weight_decay=0.01)
    for t in range(3):
        x = torch.randn(16, 48, generator=torch.Generator().manual_seed(t)).to(DEV, torch.bfloat16)
        (net(x).float() ** 2).mean().backward()
        for p, r in zip(params, refs):
            O.sgd_step(r, p.grad.reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16), 5e-2, 0.9, 0.01)
        opt.step()
        opt.zero_grad(set_to_none=True)
        torch.cuda.synchronize()
        for p, r in zip(params, refs):
            st = opt.state[p]
            assert np.array_equal(p.detach().reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16), r.param)
            assert np.array_equal(st["rho"].cpu().numpy(), r.rho)
            assert np.array_equal(st["m_codes"].cpu().numpy(), r.m)
            assert np.array_equal(st["m_scales"].cpu().view(torch.int16).numpy().view(np.uint16), r.m_scales)
