"""The step in the ablation formats (fo_adamw_step_general) against the CPU
oracle, bit for bit: every parameter format (24- and 32-bit masters, a bf16
parameter without a split, an fp32 parameter) with every state format
(companded codes, linear codes, fp32 states), fp32 and bf16 gradients, over a
ragged list and several steps.  And in the paper's own format, the general
kernel gives the same bits as the fast one."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_state_optimizer_gb300 as fo
import workloads as W
from quantized_state_optimizer_gb300 import FoTensorGeneral

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
NUMELS = [1, 33, 4096 + 17, 12345, 0, 64]


def _theta(i, n):
    g = torch.Generator().manual_seed(300 + i)
    return (torch.randn(n, generator=g) * 0.02).float()


def _grad(i, t, n, dtype):
    g = torch.Generator().manual_seed(W.grad_seed(55, i, t))
    x = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g)) * 1e-3
    return x if dtype == torch.float32 else x.to(torch.bfloat16)


class DevTensor:
    """Device buffers of one tensor in the given formats, initialised from theta."""

    def __init__(self, theta, pf, sf, grad_dtype):
        n = theta.numel()
        self.n, self.pf, self.sf = n, pf, sf
        t = theta.to(DEV)
        if pf in ("bf16_rho8", "bf16_rho16"):
            rb = 8 if pf == "bf16_rho8" else 16
            self.param = torch.empty(n, dtype=torch.bfloat16, device=DEV)
            self.rho = torch.empty(n, dtype=torch.int8 if rb == 8 else torch.int16, device=DEV)
            if n:
                fo.fo_split(t, rb, self.param, self.rho)
        elif pf == "bf16":
            self.param, self.rho = t.to(torch.bfloat16), None
        else:
            self.param, self.rho = t.clone(), None
        if sf == "f32":
            self.m = torch.zeros(n, dtype=torch.float32, device=DEV)
            self.v = torch.zeros(n, dtype=torch.float32, device=DEV)
            self.ms = self.vs = None
        else:
            self.m = torch.zeros(n, dtype=torch.int8, device=DEV)
            self.v = torch.zeros(n, dtype=torch.uint8, device=DEV)
            self.ms = torch.zeros((n + 31) // 32, dtype=torch.float16, device=DEV)
            self.vs = torch.zeros((n + 31) // 32, dtype=torch.float16, device=DEV)
        self.grad = torch.zeros(n, dtype=grad_dtype, device=DEV)

    def ft(self):
        p = lambda x: x.data_ptr() if x is not None else None  # noqa: E731
        return FoTensorGeneral(p(self.param), p(self.rho), p(self.grad), p(self.m), p(self.ms), p(self.v),
                               p(self.vs), self.n)

    def host(self):
        def bits(x):
            if x is None:
                return None
            x = x.cpu()
            if x.dtype in (torch.bfloat16, torch.float16):
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
        return {k: bits(getattr(self, k)) for k in ("param", "rho", "m", "ms", "v", "vs")}


def _oracle_state(theta, pf, sf):
    qs = sf != "f32"
    if pf == "f32":
        return O.TensorState.init(theta.numpy(), quantize_states=qs, param_dtype="f32")
    mb = {"bf16_rho8": 24, "bf16_rho16": 32, "bf16": None}[pf]
    return O.TensorState.init(theta.numpy(), master_bits=mb, quantize_states=qs)


def _same(a, b, ctx):
    if a is None and (b is None or b.size == 0):
        return
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, ctx
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.flatnonzero(a != b)
    assert bad.size == 0, f"{ctx}: {bad.size} of {a.size} differ (first {bad[:5]})"


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sf", ["companded", "linear", "f32"])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16", "bf16", "f32"])
def test_general_step_matches_oracle(pf, sf, grad_dtype):
    h = W.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05, steps=3)
    thetas = [_theta(i, n) for i, n in enumerate(NUMELS)]
    dev = [DevTensor(t, pf, sf, grad_dtype) for t in thetas]
    refs = [_oracle_state(t, pf, sf) for t in thetas]
    arr = (FoTensorGeneral * len(dev))(*[d.ft() for d in dev])
    for t in range(1, h.steps + 1):
        for i, n in enumerate(NUMELS):
            if n == 0:
                continue
            g = _grad(i, t, n, grad_dtype)
            dev[i].grad.copy_(g.to(DEV))
            gn = g.numpy() if grad_dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16)
            O.adamw_step(refs[i], gn, t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay,
                         quantize_states=sf != "f32", companded=sf == "companded")
        fo.fo_adamw_step_general(arr, pf, sf, grad_dtype, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, t)
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
            _same(got["v"], r.v, ctx + ("v",))
            if sf != "f32":
                _same(got["ms"], r.m_scales, ctx + ("m_scales",))
                _same(got["vs"], r.v_scales, ctx + ("v_scales",))


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_general_entry_equals_fo_adamw_step_in_the_papers_format(rho_bits):
    """fo_adamw_step_general in the paper's format (split master, companded
    codes) runs the pipelined kernel of fo_adamw_step through its own argument
    path: the same bits."""
    from quantized_state_optimizer_gb300.optim import FlashAdamWState
    numels = [70000, 4096 * 5 + 3, 31]
    h = W.LLAMA3_8B_HYPER
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=torch.bfloat16, device=DEV)
    pf = "bf16_rho8" if rho_bits == 8 else "bf16_rho16"
    gen = []
    for i, n in enumerate(numels):
        th = _theta(i, n)
        st.init_theta(i, th.to(DEV))
        gen.append(DevTensor(th, pf, "companded", torch.bfloat16))
    arr = (FoTensorGeneral * len(gen))(*[d.ft() for d in gen])
    for t in (1, 2, 3):
        for i, n in enumerate(numels):
            g = _grad(i, t, n, torch.bfloat16).to(DEV)
            st.grad_view(i).copy_(g)
            gen[i].grad.copy_(g)
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        fo.fo_adamw_step_general(arr, pf, "companded", torch.bfloat16, h.lr, h.beta1, h.beta2, h.eps,
                                 h.weight_decay, t)
        torch.cuda.synchronize()
        for i in range(len(numels)):
            v = st.view(i)
            d = gen[i]
            for a, b in ((v["param"], d.param), (v["rho"], d.rho), (v["m_codes"], d.m), (v["v_codes"], d.v),
                         (v["m_scales"], d.ms), (v["v_scales"], d.vs)):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (i, t)


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16"])
def test_linear_codes_split_master_pipelined(pf, grad_dtype):
    """Linear codes with a split master run in the pipelined kernel: several
    full tiles of each width (7680, 6656 and 6144 elements), ragged tails and
    heavy-tailed weights and gradients, against the oracle bit for bit."""
    h = W.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05, steps=3)
    numels = [70000, 7680 * 3, 31, 6656 * 2 + 3, 6144 * 2, (1 << 20) + 5]

    def theta_of(i, n):
        g = torch.Generator().manual_seed(800 + i)
        return (torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 2) * 0.02).float()

    thetas = [theta_of(i, n) for i, n in enumerate(numels)]
    dev = [DevTensor(t, pf, "linear", grad_dtype) for t in thetas]
    refs = [_oracle_state(t, pf, "linear") for t in thetas]
    arr = (FoTensorGeneral * len(dev))(*[d.ft() for d in dev])
    for t in range(1, h.steps + 1):
        for i, n in enumerate(numels):
            g = torch.Generator().manual_seed(W.grad_seed(57, i, t))
            # tails up to about 1e2: v stays inside fp16's range, so every
            # linear v scale is finite (an infinite one makes the next step's
            # states NaN, outside the step's preconditions)
            x = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 2) * 1e-3
            x = x if grad_dtype == torch.float32 else x.to(torch.bfloat16)
            dev[i].grad.copy_(x.to(DEV))
            gn = x.numpy() if grad_dtype == torch.float32 else x.view(torch.int16).numpy().view(np.uint16)
            O.adamw_step(refs[i], gn, t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, companded=False)
        fo.fo_adamw_step_general(arr, pf, "linear", grad_dtype, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, t)
        torch.cuda.synchronize()
        for i in range(len(numels)):
            got, r = dev[i].host(), refs[i]
            ctx = (pf, str(grad_dtype), i, t)
            for key, ref in (("param", r.param), ("rho", r.rho), ("m", r.m), ("v", r.v), ("ms", r.m_scales),
                             ("vs", r.v_scales)):
                _same(got[key], ref, ctx + (key,))


def _tie_grads(n: int, sf: str, seed: int) -> torch.Tensor:
    """fp32 gradients for one step with beta1 = 1/2, beta2 = 0 (m = g/2
    exactly, v = RN(g^2)) under which nearly every code argument lies within
    about 1e-6 of a half-integer.  Element 0 of each group of 32 is g = 2: the
    momentum scale becomes 1, the variance scale 2 (companded: fp16 of
    sqrt(4)) or 4 (linear).  Even elements tie the momentum code t = k + 1/2:
    m = t/(254 - t) (companded, the inverse softsign of t/127) or t/127
    (linear).  Odd elements tie the variance code: |g| = 2t/255 (companded:
    t = 255 sqrt(v)/2) or 2 sqrt(t/255) (linear: t = 255 v/4)."""
    rng = np.random.default_rng(seed)
    g = np.empty(n, np.float64)
    sign = rng.choice([-1.0, 1.0], n)
    k_m = rng.integers(0, 127, n) + 0.5
    k_v = rng.integers(0, 255, n) + 0.5
    m_tie = k_m / (254.0 - k_m) if sf == "companded" else k_m / 127.0
    v_tie = 2.0 * k_v / 255.0 if sf == "companded" else 2.0 * np.sqrt(k_v / 255.0)
    idx = np.arange(n)
    g[:] = np.where(idx % 2 == 0, 2.0 * m_tie, v_tie)
    g[idx % 32 == 0] = 2.0
    return torch.from_numpy((sign * g).astype(np.float32))


@pytest.mark.parametrize("sf", ["companded", "linear"])
@pytest.mark.parametrize("pf", ["bf16_rho8", "bf16_rho16", "bf16", "f32"])
def test_code_arguments_on_half_integer_ties(pf, sf):
    """Code arguments a hair from a half-integer in nearly every element: the
    kernel's certified codes cannot decide them, so every pair of every thread
    takes its codes from the definition's chain out of line; the rest of the
    step stays on the fast path.  Full tiles and a ragged tail, bit for bit
    against the oracle."""
    h = W.Hyper(lr=1e-3, beta1=0.5, beta2=0.0, eps=1e-8, weight_decay=0.05, steps=1)
    numels = [3 * 11776 + 1000, 4096]
    thetas = [_theta(10 + i, n) for i, n in enumerate(numels)]
    dev = [DevTensor(t, pf, sf, torch.float32) for t in thetas]
    refs = [_oracle_state(t, pf, sf) for t in thetas]
    arr = (FoTensorGeneral * len(dev))(*[d.ft() for d in dev])
    for i, n in enumerate(numels):
        g = _tie_grads(n, sf, 77 + i)
        dev[i].grad.copy_(g.to(DEV))
        O.adamw_step(refs[i], g.numpy(), 1, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay,
                     quantize_states=True, companded=sf == "companded")
    fo.fo_adamw_step_general(arr, pf, sf, torch.float32, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 1)
    torch.cuda.synchronize()
    for i, n in enumerate(numels):
        got, r = dev[i].host(), refs[i]
        ctx = (pf, sf, i)
        _same(got["param"], r.param, ctx + ("param",))
        if r.rho is not None:
            _same(got["rho"], r.rho, ctx + ("rho",))
        for k, rk in (("m", r.m), ("v", r.v), ("ms", r.m_scales), ("vs", r.v_scales)):
            _same(got[k], rk, ctx + (k,))
        # the construction did what it says: scales 1 and 2 (or 4), and the
        # tied codes split between the two neighbours of each half-integer
        assert np.all(r.m_scales == np.float16(1.0).view(np.uint16))
        assert np.all(r.v_scales == np.float16(2.0 if sf == "companded" else 4.0).view(np.uint16))
