"""Pins of the oracle's FlashAdamW step (page "code/flashsim/flash_adamw_sim.py",
``FlashAdamWSim.step``, Algorithm 4).

* With fp32 states and an fp32 parameter the method reduces to standard
  decoupled AdamW: compared with ``torch.optim.AdamW`` run in float64.
* From an all-zero state the first step has the closed form
  theta1 = theta0 (1 - lr wd) - lr g / (|g| + eps).
* A group whose 32 gradients are all equal keeps all codes at the top of the
  range (while its scale is a normal fp16 number), so its dequantized state is
  exactly +/- the fp16 scale: a binary64 recursion with numpy's float16
  rounding predicts every step.
* Zero gradients leave zero states at zero and only decay theta.
"""

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests.test_oracle_split import round_to_master24_f64

H = W.SINGLE_TENSOR_HYPER
U = 2.0 ** -24  # unit roundoff of binary32


def _f16(x):
    return np.float64(np.float16(x))


def test_unquantized_fp32_reduces_to_torch_adamw():
    n = 4096 + 17
    theta0 = W.single_tensor_theta(n).numpy()
    st = O.TensorState.init(theta0, quantize_states=False, param_dtype="f32")
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=H.lr, betas=(H.beta1, H.beta2), eps=H.eps,
                            weight_decay=H.weight_decay, foreach=False)
    for t in range(1, 11):
        g = W.single_tensor_grad(t, n).numpy()
        O.adamw_step(st, g, t, H.lr, H.beta1, H.beta2, H.eps, H.weight_decay, quantize_states=False)
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        ref = p.detach().numpy()
        # a few binary32 roundings of |theta| (~0.02-0.1) per step
        assert np.max(np.abs(st.param - ref)) <= 8 * U * 0.1 * t
        s = opt.state[p]
        mr, vr = s["exp_avg"].numpy(), s["exp_avg_sq"].numpy()
        assert np.max(np.abs(st.m - mr)) <= 1e-5 * np.max(np.abs(mr))
        assert np.max(np.abs(st.v - vr)) <= 1e-5 * np.max(np.abs(vr))


def test_decoupled_decay_multiplies_the_old_theta_first():
    """The page's step decays theta before the update (as torch's AdamW does).
    With lr wd large (lr 0.1, wd 0.5) the other order, decay after the update,
    lands lr wd |delta| away: on the first step |delta| = lr |g|/(|g| + eps)
    ~ lr, i.e. 5e-3 for every element, far above the binary32 error of
    either.  The oracle must match torch's order on every step, and lie that
    far from the other order on the first."""
    n = 1000
    g0 = torch.Generator().manual_seed(21)
    theta0 = (torch.randn(n, generator=g0) * 0.02).numpy().astype(np.float32)
    lr, b1, b2, eps, wd = 0.1, 0.9, 0.999, 1e-8, 0.5
    st = O.TensorState.init(theta0, quantize_states=False, param_dtype="f32")
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    for t in range(1, 6):
        g = (torch.randn(n, generator=g0) * 1e-3).numpy().astype(np.float32)
        O.adamw_step(st, g, t, lr, b1, b2, eps, wd, quantize_states=False)
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        assert np.max(np.abs(st.param - p.detach().numpy())) <= 1e-5
        if t == 1:
            g64 = g.astype(np.float64)
            after = (theta0 - lr * g64 / (np.abs(g64) + eps)) * (1 - lr * wd)
            assert np.min(np.abs(st.param - after)) >= 4e-3


@pytest.mark.parametrize("master_bits", [24, 32])
def test_first_step_closed_form(master_bits):
    n = W.SINGLE_TENSOR_NUMEL
    theta0 = W.single_tensor_theta(n).numpy()
    st = O.TensorState.init(theta0, master_bits=master_bits)
    th0 = st.theta().astype(np.float64)
    g = W.single_tensor_grad(1, n).numpy()
    O.adamw_step(st, g, 1, H.lr, H.beta1, H.beta2, H.eps, H.weight_decay)
    g64 = g.astype(np.float64)
    delta = H.lr * g64 / (np.abs(g64) + H.eps)
    th1 = th0 * (1 - H.lr * H.weight_decay) - delta
    got = st.theta().astype(np.float64)
    # binary32 roundings scale with the operands, not with the (possibly cancelled) result
    fp32_err = 8 * U * (np.abs(th0) + np.abs(delta))
    master_err = 2.0 ** -16 * np.abs(th1) if master_bits == 24 else 0.0
    assert np.all(np.abs(got - th1) <= master_err * (1 + 1e-6) + fp32_err)
    # the new states dequantize to (1-b1) g and (1-b2) g^2 within a code step
    m = O.dequantize(st.m, st.m_scales, "momentum").astype(np.float64)
    sm = np.repeat(O.f16_bits_to_f32(st.m_scales).astype(np.float64), 32)[:n]
    xm = (1 - H.beta1) * g64
    assert np.all(np.abs(m - xm) <= sm / 127 * 1.001 + np.maximum(0, np.abs(xm) - sm) + 1e-12)
    v = O.dequantize(st.v, st.v_scales, "variance").astype(np.float64)
    sv = np.repeat(O.f16_bits_to_f32(st.v_scales).astype(np.float64), 32)[:n]
    rv = np.sqrt(1 - H.beta2) * np.abs(g64)
    assert np.all(np.abs(np.sqrt(v) - rv) <= sv * 0.5 / 255 * 1.001 + np.maximum(0, rv - sv) + 1e-12)


@pytest.mark.parametrize("master_bits", [24, 32])
def test_first_step_with_linear_codes(master_bits):
    """Linear codes (companded=False): the first step's theta equals the
    fp32-state step's bit for bit (both start from zero states), and the
    stored codes are that step's exact m and v quantized with the
    MOMENTUM_LINEAR / VARIANCE_LINEAR specs (v itself, no square root)."""
    n = W.SINGLE_TENSOR_NUMEL
    theta0 = W.single_tensor_theta(n).numpy()
    g = W.single_tensor_grad(1, n).numpy()
    st = O.TensorState.init(theta0, master_bits=master_bits)
    ref = O.TensorState.init(theta0, master_bits=master_bits, quantize_states=False)
    O.adamw_step(st, g, 1, H.lr, H.beta1, H.beta2, H.eps, H.weight_decay, companded=False)
    O.adamw_step(ref, g, 1, H.lr, H.beta1, H.beta2, H.eps, H.weight_decay, quantize_states=False)
    assert np.array_equal(st.param, ref.param) and np.array_equal(st.rho, ref.rho)
    # the fp32 states are the definition's first moments, each op rounded once
    assert np.array_equal(ref.m, np.float32(1 - H.beta1) * g)
    assert np.array_equal(ref.v, (np.float32(1 - H.beta2) * g) * g)
    mc, ms = O.quantize(ref.m, "momentum_linear")
    vc, vs = O.quantize(ref.v, "variance_linear")
    assert np.array_equal(st.m, mc) and np.array_equal(st.m_scales, ms)
    assert np.array_equal(st.v, vc) and np.array_equal(st.v_scales, vs)


@pytest.mark.parametrize("master_bits", [24, 32])
def test_constant_gradient_groups_closed_form(master_bits):
    rng = np.random.default_rng(5)
    G, T = 64, 8
    # magnitudes keep (1-b1)|c| and sqrt(1-b2)|c| above the fp16 normal limit 2^-14
    c = (np.sign(rng.standard_normal(G)) * 10.0 ** rng.uniform(-2.5, -0.5, G)).astype(np.float32)
    grad = np.repeat(c, 32)
    theta0 = (rng.standard_normal(G * 32) * 0.02).astype(np.float32)
    st = O.TensorState.init(theta0, master_bits=master_bits)
    th = st.theta().astype(np.float64)
    mq = np.zeros(G)  # dequantized state carried between steps
    vq = np.zeros(G)
    c64 = c.astype(np.float64)
    b1, b2, lr, eps, wd = 0.9, 0.999, 1e-3, 1e-8, 0.01
    for t in range(1, T + 1):
        O.adamw_step(st, grad, t, lr, b1, b2, eps, wd)
        m = b1 * mq + (1 - b1) * c64
        v = b2 * vq + (1 - b2) * c64 * c64
        upd = lr * (m / (1 - b1 ** t)) / (np.sqrt(v / (1 - b2 ** t)) + eps)
        pred = th * (1 - lr * wd) - np.repeat(upd, 32)
        if master_bits == 24:
            pred = round_to_master24_f64(pred)
        # requantized state: top code, fp16 scale of the (common) value
        sm = np.array([_f16(abs(x)) for x in m])
        sv = np.array([_f16(np.sqrt(x)) for x in v])
        got_sm = O.f16_bits_to_f32(st.m_scales).astype(np.float64)
        got_sv = O.f16_bits_to_f32(st.v_scales).astype(np.float64)
        # binary32 vs binary64 may straddle an fp16 rounding boundary: one fp16 step
        assert np.all(np.abs(got_sm - sm) <= sm * 2.0 ** -10), t
        assert np.all(np.abs(got_sv - sv) <= sv * 2.0 ** -10), t
        assert np.all(st.m.reshape(G, 32) == (np.sign(c) * 127).astype(np.int8)[:, None]), t
        assert np.all(st.v == 255), t
        mq = np.sign(m) * got_sm
        vq = got_sv * got_sv
        got = st.theta().astype(np.float64)
        fp32_err = 8 * U * (np.abs(th) + np.repeat(np.abs(upd), 32))
        master_err = 2.0 ** -15 * np.abs(pred) if master_bits == 24 else 0.0
        assert np.all(np.abs(got - pred) <= master_err + fp32_err), t
        th = got  # carry the oracle's own master forward (rounding is pinned per step)


def test_zero_gradient_keeps_zero_state_and_decays_theta():
    n = 1000
    theta0 = W.single_tensor_theta(n).numpy()
    st = O.TensorState.init(theta0, master_bits=32)
    c = 1 - H.lr * 0.1
    for t in range(1, 6):
        O.adamw_step(st, np.zeros(n, np.float32), t, H.lr, H.beta1, H.beta2, H.eps, 0.1)
        assert np.all(st.m == 0) and np.all(st.v == 0)
        assert np.all(st.m_scales == 0) and np.all(st.v_scales == 0)
        ref = theta0.astype(np.float64) * c ** t
        assert np.all(np.abs(st.theta() - ref) <= 2 * t * U * np.abs(ref))


def test_bf16_grads_equal_their_fp32_widening():
    n = 4096
    theta0 = W.single_tensor_theta(n).numpy()
    g32 = W.single_tensor_grad(1, n).numpy()
    gb = O.f32_to_bf16_rne_bits(g32)
    st_a = O.TensorState.init(theta0, master_bits=32)
    st_b = O.TensorState.init(theta0, master_bits=32)
    O.adamw_step(st_a, gb, 1, H.lr, H.beta1, H.beta2, H.eps, 0.0)
    O.adamw_step(st_b, (gb.astype(np.uint32) << 16).view(np.float32), 1, H.lr, H.beta1, H.beta2,
                 H.eps, 0.0)
    for a, b in ((st_a.param, st_b.param), (st_a.rho, st_b.rho), (st_a.m, st_b.m), (st_a.v, st_b.v)):
        assert np.array_equal(a, b)


def test_quantized_trajectory_tracks_fp64_adamw():
    """Loose: 8-bit states move the trajectory by a small fraction of the total
    displacement; a dropped term or a wrong sign moves it by O(1) of it."""
    n = W.SINGLE_TENSOR_NUMEL
    theta0 = W.single_tensor_theta(n).numpy()
    st = O.TensorState.init(theta0, master_bits=24)
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=H.lr, betas=(H.beta1, H.beta2), eps=H.eps,
                            weight_decay=H.weight_decay, foreach=False)
    for t in range(1, H.steps + 1):
        g = W.single_tensor_grad(t, n).numpy()
        O.adamw_step(st, g, t, H.lr, H.beta1, H.beta2, H.eps, H.weight_decay)
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
    ref = p.detach().numpy()
    disp = np.abs(ref - theta0).mean()
    err = np.abs(st.theta() - ref).mean()
    assert err < 0.05 * disp, (err, disp)


def test_step_argument_errors():
    st = O.TensorState.init(np.zeros(8, np.float32))
    with pytest.raises(RuntimeError):
        O.adamw_step(st, np.zeros(8, np.float32), 0, 1e-3, 0.9, 0.999, 1e-8, 0.0)
