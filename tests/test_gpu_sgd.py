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


# ---------------------------------------------------------------------------
# The paper's format (bf16 theta' + int8/int16 rho, companded momentum codes)
# runs in the pipelined kernel: full tiles through the bulk-copy stages with
# certified codes, ragged tails with ordinary loads.  Its tiles hold 7680
# elements (bf16 grads, int8 rho), 6656 (bf16, int16 rho; fp32, int8 rho) or
# 6144 (fp32, int16 rho).

def _run_sgd(numels, pf, grad_dtype, lr, mu, wd, steps, grad_fn=None, theta_fn=None, sf="companded"):
    thetas = [theta_fn(i, n) if theta_fn else _theta(i, n) for i, n in enumerate(numels)]
    dev = [DevTensor(t, pf, sf, grad_dtype) for t in thetas]
    refs = [_oracle_state(t, pf, sf) for t in thetas]
    arr = (FoTensorGeneral * len(dev))(*[d.ft() for d in dev])
    for k in range(len(arr)):
        arr[k].v = None
        arr[k].v_scales = None
    for t in range(1, steps + 1):
        for i, n in enumerate(numels):
            if n == 0:
                continue
            g = grad_fn(i, t, n) if grad_fn else _grad(i, t, n, grad_dtype)
            g = g if grad_dtype == torch.float32 else g.to(torch.bfloat16)
            dev[i].grad.copy_(g.to(DEV))
            gn = g.numpy() if grad_dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16)
            O.sgd_step(refs[i], gn, lr, mu, wd, companded=sf == "companded")
        fo.fo_sgd_step(arr, pf, sf, grad_dtype, lr, mu, wd)
        torch.cuda.synchronize()
        for i, n in enumerate(numels):
            if n == 0:
                continue
            got, r = dev[i].host(), refs[i]
            ctx = (pf, str(grad_dtype), mu, wd, i, n, t)
            _same(got["param"], r.param, ctx + ("param",))
            _same(got["rho"], r.rho, ctx + ("rho",))
            _same(got["m"], r.m, ctx + ("m",))
            _same(got["ms"], r.m_scales, ctx + ("m_scales",))


@pytest.mark.parametrize("sf", ["companded", "linear"])
@pytest.mark.parametrize("mu,wd", [(0.9, 0.01), (0.9, 0.0), (0.0, 0.0)])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16"])
def test_sgd_fast_kernel_full_tiles(pf, grad_dtype, mu, wd, sf):
    numels = [70000, 7680 * 3, 31, 6656 * 2 + 3, 0, 6144 * 2, 100003]
    _run_sgd(numels, pf, grad_dtype, 1e-2, mu, wd, 3, sf=sf)


def test_sgd_more_tensors_than_one_launch():
    rng = np.random.default_rng(1)
    numels = [int(x) for x in rng.integers(1, 9000, fo.fo_max_tensors_per_launch() + 23)]
    _run_sgd(numels, "bf16_rho8", torch.bfloat16, 1e-2, 0.9, 0.01, 2)


@pytest.mark.parametrize("sf", ["companded", "linear"])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16"])
def test_sgd_volume_heavy_tailed(pf, sf):
    """Millions of elements, weights and gradients over many orders of magnitude."""
    def theta_fn(i, n):
        g = torch.Generator().manual_seed(700 + i)
        return (torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 2) * 0.02).float()

    def grad_fn(i, t, n):
        g = torch.Generator().manual_seed(W.grad_seed(88, i, t))
        return torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 3) * 1e-3

    _run_sgd([(1 << 22) + 5, 3 * (1 << 20)], pf, torch.bfloat16, 1e-2, 0.9, 0.05, 4, grad_fn, theta_fn, sf=sf)


def test_sgd_half_integer_codes_leave_every_certificate_open():
    """On the first step the buffer is the gradient itself.  Gradients chosen
    so that every element but the group maximum 1.0 has a code argument
    127 * 2y/(1+y) next to a half-integer k + 1/2 (y = (k + 1/2)/(254 - k - 1/2),
    rounded to fp32) leave nearly every code certificate open, so nearly every
    thread finishes through the exact path."""
    k = np.arange(31) * 4 + 0.5
    y = (k / (254.0 - k)).astype(np.float32)
    group = np.concatenate([[np.float32(1.0)], y]).astype(np.float32)

    def grad_fn(i, t, n):
        if t == 1:
            reps = (n + 31) // 32
            sign = np.where(np.arange(reps * 32) % 3 == 0, -1.0, 1.0).astype(np.float32)
            return torch.from_numpy((np.tile(group, reps) * sign)[:n].copy())
        return _grad(i, t, n, torch.float32)

    _run_sgd([6656 * 3 + 45, 6144 * 2], "bf16_rho8", torch.float32, 1e-2, 0.9, 0.0, 2, grad_fn)
    _run_sgd([6144 * 3 + 45], "bf16_rho16", torch.float32, 1e-2, 0.9, 0.0, 2, grad_fn)
