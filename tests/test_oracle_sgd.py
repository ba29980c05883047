"""Pins of the oracle's FlashSGD step (the reading of fo_oracle.h [B]: SGD with
momentum as torch.optim.SGD, momentum buffer stored like FlashAdamW's m,
master weight split as in FlashAdamW) against references outside the oracle:
torch.optim.SGD in binary64, closed forms, special cases."""

import numpy as np
import pytest
import torch

import oracle as O


def _sgd64(theta0, grads, lr, mu, wd):
    """torch.optim.SGD (dampening 0, no Nesterov) in binary64 on CPU."""
    p = torch.nn.Parameter(torch.tensor(theta0, dtype=torch.float64))
    opt = torch.optim.SGD([p], lr=lr, momentum=mu, weight_decay=wd, foreach=False)
    out = []
    for g in grads:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        out.append(p.detach().numpy().copy())
    return out


def _f32_state(theta):
    return O.TensorState.init(theta, quantize_states=False, param_dtype="f32")


@pytest.mark.parametrize("mu,wd", [(0.9, 0.0), (0.9, 0.01), (0.0, 0.1), (0.5, 0.0)])
def test_fp32_states_reduce_to_torch_sgd(mu, wd):
    rng = np.random.default_rng(3)
    theta0 = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(1000) * 1e-3).astype(np.float32) for _ in range(6)]
    st = _f32_state(theta0)
    ref = _sgd64(theta0.astype(np.float64), [g.astype(np.float64) for g in grads], 0.05, mu, wd)
    for t, g in enumerate(grads):
        O.sgd_step(st, g, 0.05, mu, wd, quantize_states=False)
        np.testing.assert_allclose(st.param, ref[t], rtol=2e-6, atol=1e-9)


def test_constant_gradient_closed_form():
    """buf_t = c (1 + mu + ... + mu^(t-1)), theta_t = theta_0 - lr sum_k buf_k."""
    n, c, lr, mu = 96, np.float32(0.0625), 0.125, 0.5
    st = _f32_state(np.ones(n, np.float32))
    buf, theta = 0.0, 1.0
    for _ in range(8):
        O.sgd_step(st, np.full(n, c, np.float32), lr, mu, 0.0, quantize_states=False)
        buf = mu * buf + float(c)
        theta = theta - lr * buf
        np.testing.assert_allclose(st.m, buf, rtol=1e-6)
        np.testing.assert_allclose(st.param, theta, rtol=1e-6)


@pytest.mark.parametrize("master_bits", [24, 32])
def test_momentum_zero_is_plain_sgd_in_every_state_format(master_bits):
    """With mu = 0 the stored buffer is never read back: theta follows plain SGD
    whatever the state format, and the buffer codes are the quantized gradient."""
    rng = np.random.default_rng(5)
    theta0 = (rng.standard_normal(4096 + 11) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(theta0.size) * 1e-3).astype(np.float32) for _ in range(3)]
    a = O.TensorState.init(theta0, master_bits=master_bits)
    b = O.TensorState.init(theta0, master_bits=master_bits, quantize_states=False)
    for g in grads:
        O.sgd_step(a, g, 1e-2, 0.0, 0.0)
        O.sgd_step(b, g, 1e-2, 0.0, 0.0, quantize_states=False)
        assert np.array_equal(a.param, b.param) and np.array_equal(a.rho, b.rho)
        codes, scales = O.quantize(g, "momentum")
        assert np.array_equal(a.m, codes) and np.array_equal(a.m_scales, scales)


def test_quantized_momentum_tracks_fp64_sgd():
    rng = np.random.default_rng(9)
    theta0 = (rng.standard_normal(8192) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(8192) * 1e-3).astype(np.float32) for _ in range(10)]
    st = O.TensorState.init(theta0, master_bits=32)
    ref = _sgd64(theta0.astype(np.float64), [g.astype(np.float64) for g in grads], 1e-2, 0.9, 0.0)
    for t, g in enumerate(grads):
        O.sgd_step(st, g, 1e-2, 0.9, 0.0)
        moved = np.abs(ref[t] - theta0.astype(np.float64))
        err = np.abs(st.theta().astype(np.float64) - ref[t])
        # quantized momentum: error a small fraction of the distance travelled
        assert np.median(err / np.maximum(moved, 1e-12)) < 0.02, t


def test_zero_gradient_decays_theta_with_coupled_weight_decay():
    """g = 0, mu = 0: theta_{t+1} = theta_t (1 - lr wd) up to fp32 rounding."""
    theta0 = np.linspace(-1, 1, 256, dtype=np.float32)
    st = _f32_state(theta0)
    expect = theta0.astype(np.float64)
    for _ in range(4):
        O.sgd_step(st, np.zeros(256, np.float32), 0.1, 0.0, 0.5, quantize_states=False)
        expect = expect * (1 - 0.1 * 0.5)
        np.testing.assert_allclose(st.param, expect, rtol=1e-6, atol=1e-7)


def test_bad_arguments():
    st = _f32_state(np.ones(4, np.float32))
    st.param_kind = 9
    with pytest.raises(RuntimeError):
        O.sgd_step(st, np.zeros(4, np.float32), 0.1, 0.9, 0.0, quantize_states=False)


@pytest.mark.parametrize("master_bits", [24, 32])
def test_momentum_zero_with_linear_codes(master_bits):
    """Linear momentum codes: with mu = 0 theta follows plain SGD exactly as
    with fp32 states, and the stored buffer is that step's buffer (g + wd theta,
    which the fp32-state run holds exactly) quantized with the MOMENTUM_LINEAR
    spec."""
    rng = np.random.default_rng(13)
    theta0 = (rng.standard_normal(4096 + 5) * 0.02).astype(np.float32)
    a = O.TensorState.init(theta0, master_bits=master_bits)
    b = O.TensorState.init(theta0, master_bits=master_bits, quantize_states=False)
    for _ in range(3):
        g = (rng.standard_normal(theta0.size) * 1e-3).astype(np.float32)
        O.sgd_step(a, g, 1e-2, 0.0, 0.01, companded=False)
        O.sgd_step(b, g, 1e-2, 0.0, 0.01, quantize_states=False)
        assert np.array_equal(a.param, b.param) and np.array_equal(a.rho, b.rho)
        codes, scales = O.quantize(b.m.astype(np.float32), "momentum_linear")
        assert np.array_equal(a.m, codes) and np.array_equal(a.m_scales, scales)
