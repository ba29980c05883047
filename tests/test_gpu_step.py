"""GPU parity of the fused multi-tensor FlashAdamW step against the CPU oracle.

Both sides start from the same seeded fp32 master weights and zero states,
split them independently, and then take the same seeded gradients step after
step; theta', rho, codes and scales must stay identical bit for bit (which
implies the looser targets: all codes within +/-1, theta within 1e-6).

The full-size Llama lists are checked on sampled groups: every group evolves
independently of all others, so the oracle carries a fixed sample of groups
through all steps and is compared with the same groups of the GPU run.
"""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_state_optimizer_gb300 as fo
import workloads as W
from quantized_state_optimizer_gb300.optim import FlashAdamW, FlashAdamWState

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _bits16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def gpu_view_np(st: FlashAdamWState, i: int) -> dict:
    v = st.view(i)
    return {"param": _bits16(v["param"]), "rho": v["rho"].cpu().numpy(),
            "m": v["m_codes"].cpu().numpy(), "m_scales": _bits16(v["m_scales"]),
            "v": v["v_codes"].cpu().numpy(), "v_scales": _bits16(v["v_scales"])}


def ref_np(r: O.TensorState) -> dict:
    return {"param": r.param, "rho": r.rho, "m": r.m, "m_scales": r.m_scales, "v": r.v,
            "v_scales": r.v_scales}


def assert_same(got: dict, ref: dict, ctx):
    for k in ("param", "rho", "m", "m_scales", "v", "v_scales"):
        a, b = np.asarray(got[k]), np.asarray(ref[k])
        assert a.shape == b.shape, (ctx, k, a.shape, b.shape)
        if not np.array_equal(a, b):
            bad = np.flatnonzero(a != b)
            raise AssertionError(f"{ctx}: {k} differs at {bad.size} of {a.size} (first {bad[:5]})")


def tolerance_report(got: dict, ref: dict, master_bits: int) -> dict:
    """The looser parity targets: code agreement, codes within +/-1, theta rel. error."""
    out = {}
    for k in ("m", "v"):
        d = np.abs(got[k].astype(int) - ref[k].astype(int))
        out[k + "_identical"] = float(np.mean(d == 0))
        out[k + "_within1"] = float(np.mean(d <= 1))
    tg = O.reconstruct(got["param"], got["rho"], master_bits).astype(np.float64)
    tr = O.reconstruct(ref["param"], ref["rho"], master_bits).astype(np.float64)
    nz = tr != 0
    out["theta_max_rel_err"] = float(np.max(np.abs(tg[nz] - tr[nz]) / np.abs(tr[nz]))) if nz.any() else 0.0
    return out


def _grad(i: int, t: int, n: int, dtype) -> torch.Tensor:
    g = torch.Generator().manual_seed(W.grad_seed(99, i, t))
    x = torch.randn(n, generator=g) * 1e-3
    return x if dtype == torch.float32 else x.to(torch.bfloat16)


def run_small(numels, rho_bits, grad_dtype, hyper: W.Hyper, steps: int, theta_fn=None):
    mb = 24 if rho_bits == 8 else 32
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=grad_dtype, device=DEV)
    refs = []
    for i, n in enumerate(numels):
        theta = theta_fn(i, n) if theta_fn else torch.randn(n, generator=torch.Generator().manual_seed(i)) * 0.02
        if n:
            st.init_theta(i, theta.to(DEV))
        refs.append(O.TensorState.init(theta.numpy(), master_bits=mb))
    for t in range(1, steps + 1):
        for i, n in enumerate(numels):
            if n == 0:
                continue
            g = _grad(i, t, n, grad_dtype)
            st.grad_view(i).copy_(g.to(DEV))
            gn = g.numpy() if grad_dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16)
            O.adamw_step(refs[i], gn, t, hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay)
        st.step(t, hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay)
        torch.cuda.synchronize()
        for i, n in enumerate(numels):
            if n:
                assert_same(gpu_view_np(st, i), ref_np(refs[i]), (numels[i], rho_bits, grad_dtype, t))
    return st, refs


def test_single_tensor_65553_fp32_grads_10_steps():
    """One flat tensor of 2^16+17 parameters, fp32 grads, 24-bit master, 10 steps."""
    n = W.SINGLE_TENSOR_NUMEL
    h = W.SINGLE_TENSOR_HYPER
    st = FlashAdamWState([n], rho_bits=8, grad_dtype=torch.float32, device=DEV)
    theta = W.single_tensor_theta(n)
    st.init_theta(0, theta.to(DEV))
    ref = O.TensorState.init(theta.numpy(), master_bits=24)
    for t in range(1, h.steps + 1):
        g = W.single_tensor_grad(t, n)
        st.grad_view(0).copy_(g.to(DEV))
        O.adamw_step(ref, g.numpy(), t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        torch.cuda.synchronize()
        got = gpu_view_np(st, 0)
        assert_same(got, ref_np(ref), ("single", t))
    rep = tolerance_report(got, ref_np(ref), 24)
    assert rep["m_identical"] == 1.0 and rep["v_identical"] == 1.0 and rep["theta_max_rel_err"] == 0.0


@pytest.mark.parametrize("rho_bits", [8, 16])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_mixed_ragged_list(rho_bits, grad_dtype, wd):
    numels = [1, 31, 33, 4096, 4097, 0, 16, 100003, 65536, 8191]
    h = W.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd, steps=3)
    run_small(numels, rho_bits, grad_dtype, h, 3)


def test_more_tensors_than_one_launch():
    rng = np.random.default_rng(0)
    count = fo.fo_max_tensors_per_launch() + 57
    numels = [int(x) for x in rng.integers(1, 300, count)]
    run_small(numels, 8, torch.bfloat16, W.LLAMA3_8B_HYPER, 2)


def test_edge_values_in_state():
    """Heavy-tailed master weights (huge, tiny, subnormal, zero) and large gradients."""
    def theta_fn(i, n):
        g = torch.Generator().manual_seed(100 + i)
        x = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 8)
        x[::7] = 0.0
        x[3::11] = 1e-39
        return x.float()
    run_small([4096 + 5, 1000], 8, torch.float32, W.SINGLE_TENSOR_HYPER, 3, theta_fn)
    run_small([4096 + 5, 1000], 16, torch.float32, W.SINGLE_TENSOR_HYPER, 3, theta_fn)


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_volume_heavy_tailed_parity(rho_bits):
    """Millions of elements with gradients and weights spread over many orders
    of magnitude, so that uncertain codes and uncertain 24-bit masters (the
    exact fallbacks of the kernel) occur thousands of times per step."""
    numels = [(1 << 22) + 7, 3 * (1 << 20)]
    mb = 24 if rho_bits == 8 else 32
    h = W.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05, steps=4)
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=torch.bfloat16, device=DEV)
    refs = []
    for i, n in enumerate(numels):
        gen = torch.Generator().manual_seed(500 + i)
        theta = torch.randn(n, generator=gen) * torch.exp(torch.randn(n, generator=gen) * 2) * 0.02
        st.init_theta(i, theta.to(DEV))
        refs.append(O.TensorState.init(theta.numpy(), master_bits=mb))
    for t in range(1, h.steps + 1):
        for i, n in enumerate(numels):
            gen = torch.Generator().manual_seed(W.grad_seed(77, i, t))
            g = (torch.randn(n, generator=gen) * torch.exp(torch.randn(n, generator=gen) * 3) * 1e-3).to(torch.bfloat16)
            st.grad_view(i).copy_(g.to(DEV))
            O.adamw_step(refs[i], g.view(torch.int16).numpy().view(np.uint16), t, h.lr, h.beta1, h.beta2,
                         h.eps, h.weight_decay)
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        torch.cuda.synchronize()
        for i in range(len(numels)):
            assert_same(gpu_view_np(st, i), ref_np(refs[i]), ("volume", rho_bits, i, t))


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_groups_with_subnormal_scales_beside_normal_ones(rho_bits):
    """Each group of 32 gets its own gradient magnitude, from 1e-9 to 1e-2:
    tiny groups have subnormal or zero fp16 scales (their code arguments can
    pass the code range and need the clamps), the others normal ones (the
    clamp-free form), side by side in every warp."""
    numels = [7680 * 2 + 4096 + 96, 33 * 32 + 5]
    h = W.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, steps=3)
    mb = 24 if rho_bits == 8 else 32
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=torch.bfloat16, device=DEV)
    refs = []
    for i, n in enumerate(numels):
        theta = torch.randn(n, generator=torch.Generator().manual_seed(40 + i)) * 0.02
        st.init_theta(i, theta.to(DEV))
        refs.append(O.TensorState.init(theta.numpy(), master_bits=mb))
    for t in range(1, h.steps + 1):
        for i, n in enumerate(numels):
            gen = torch.Generator().manual_seed(W.grad_seed(91, i, t))
            groups = (n + 31) // 32
            mag = 10.0 ** -torch.randint(2, 10, (groups,), generator=gen).double()
            g = (torch.randn(n, generator=gen).double() * mag.repeat_interleave(32)[:n]).float().to(torch.bfloat16)
            st.grad_view(i).copy_(g.to(DEV))
            O.adamw_step(refs[i], g.view(torch.int16).numpy().view(np.uint16), t, h.lr, h.beta1, h.beta2,
                         h.eps, h.weight_decay)
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        torch.cuda.synchronize()
        for i in range(len(numels)):
            got = gpu_view_np(st, i)
            assert_same(got, ref_np(refs[i]), ("subnormal scales", rho_bits, i, t))
    # both kinds of scale occurred
    ms = np.abs(st.m_scales.float().cpu().numpy())
    assert np.any((ms > 0) & (ms < 2.0 ** -14)) and np.any(ms >= 2.0 ** -14)


def test_checkpoint_resume_is_bit_identical():
    numels = [5000, 4096, 77]
    h = W.TINYLLAMA_HYPER

    def make():
        st = FlashAdamWState(numels, rho_bits=16, grad_dtype=torch.bfloat16, device=DEV)
        for i, n in enumerate(numels):
            st.init_theta(i, (torch.randn(n, generator=torch.Generator().manual_seed(i)) * 0.02).to(DEV))
        return st

    def run(st, t0, t1):
        for t in range(t0, t1 + 1):
            for i, n in enumerate(numels):
                st.grad_view(i).copy_(_grad(i, t, n, torch.bfloat16).to(DEV))
            st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)

    a = make()
    run(a, 1, 10)
    b = make()
    run(b, 1, 5)
    sd = b.state_dict()
    c = make()
    c.load_state_dict(sd)
    run(c, 6, 10)
    torch.cuda.synchronize()
    for k in ("param", "rho", "m_codes", "m_scales", "v_codes", "v_scales"):
        assert torch.equal(getattr(a, k).view(torch.uint8) if getattr(a, k).dtype != torch.uint8 else getattr(a, k),
                           getattr(c, k).view(torch.uint8) if getattr(c, k).dtype != torch.uint8 else getattr(c, k)), k


@pytest.mark.parametrize("n_chunks", [1, 3, 8])
def test_step_from_host_matches_device_step(n_chunks):
    """The host-fed step (chunked uploads, launches and downloads on three
    streams) leaves the same state as device steps on the same gradients, and
    the host copy of theta' equals the device one after every step."""
    numels = [70000, 33, 4096 * 3, 0, 12345, 9000, 1]
    h = W.LLAMA3_8B_HYPER

    def make():
        st = FlashAdamWState(numels, rho_bits=8, grad_dtype=torch.bfloat16, device=DEV)
        for i, n in enumerate(numels):
            if n:
                st.init_theta(i, (torch.randn(n, generator=torch.Generator().manual_seed(i)) * 0.02).to(DEV))
        return st

    a, b = make(), make()
    host_grad = torch.empty(b.grad.numel(), dtype=b.grad.dtype, pin_memory=True)
    host_param = torch.empty(b.param.numel(), dtype=b.param.dtype, pin_memory=True)
    for t in range(1, 5):
        for i, n in enumerate(numels):
            if n:
                a.grad_view(i).copy_(_grad(i, t, n, torch.bfloat16).to(DEV))
        host_grad.copy_(a.grad.cpu())
        a.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        b.step_from_host(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, host_grad, host_param,
                         n_chunks=n_chunks)
        torch.cuda.synchronize()
        for k in ("param", "rho", "m_codes", "m_scales", "v_codes", "v_scales"):
            x, y = getattr(a, k), getattr(b, k)
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), (k, t)
        assert torch.equal(host_param.view(torch.int16), b.param.cpu().view(torch.int16)), t


def test_torch_optimizer_front_end_matches_oracle():
    torch.manual_seed(0)
    shapes = [(64, 33), (4097,), (7,)]
    params = [torch.nn.Parameter((torch.randn(s) * 0.02).to(torch.bfloat16).to(DEV)) for s in shapes]
    refs = [O.TensorState.init(p.detach().float().cpu().numpy().reshape(-1), master_bits=24) for p in params]
    opt = FlashAdamW(params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    for t in range(1, 4):
        for i, p in enumerate(params):
            g = _grad(i, t, p.numel(), torch.bfloat16)
            p.grad = g.reshape(p.shape).to(DEV)
            O.adamw_step(refs[i], g.view(torch.int16).numpy().view(np.uint16), t, 1e-3, 0.9, 0.999, 1e-8, 0.01)
        opt.step()
    torch.cuda.synchronize()
    for p, r in zip(params, refs):
        s = opt.state[p]
        got = {"param": _bits16(p.detach().reshape(-1)), "rho": s["rho"].cpu().numpy(),
               "m": s["m_codes"].cpu().numpy(), "m_scales": _bits16(s["m_scales"]),
               "v": s["v_codes"].cpu().numpy(), "v_scales": _bits16(s["v_scales"])}
        assert_same(got, ref_np(r), "FlashAdamW")


def test_zero_initialized_weights():
    """theta = 0: the new theta is -delta itself, so the master carries every
    bit of the update (no bits of an old theta to round into)."""
    numels = [7680 * 4, 7680 * 2 + 33]
    run_small(numels, 8, torch.bfloat16, W.LLAMA3_8B_HYPER, 3, theta_fn=lambda i, n: torch.zeros(n))


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_cancelling_update(rho_bits):
    """theta = lr sign(g): the first step's update nearly cancels theta, so the
    new theta is a small difference of two close values (tiny, subnormal-free
    results whose low bits all come from delta)."""
    h = W.LLAMA3_8B_HYPER
    numels = [7680 * 3 + 17]

    def theta_fn(i, n):
        return torch.sign(_grad(i, 1, n, torch.bfloat16).float()) * h.lr

    run_small(numels, rho_bits, torch.bfloat16, h, 2, theta_fn)


def test_device_status_clear_after_steps():
    fo.fo_device_status()  # clear anything left by earlier tests
    run_small([20000, 7680 * 3, 7680 + 5], 8, torch.bfloat16, W.LLAMA3_8B_HYPER, 2)
    torch.cuda.synchronize()
    assert fo.fo_device_status() == 0


def test_argument_errors_through_binding():
    st = FlashAdamWState([100], rho_bits=8, device=DEV)
    with pytest.raises(fo.FoError, match="INVALID_ARG"):
        st.step(0, 1e-3, 0.9, 0.999, 1e-8, 0.0)
    with pytest.raises(fo.FoError, match="INVALID_ARG"):
        st.step(1, 1e-3, 1.0, 0.999, 1e-8, 0.0)
    arr = st.fo_tensors()
    bad = (fo.FoTensor * 2)(arr[0], arr[0])  # the same buffers twice
    with pytest.raises(fo.FoError, match="ALIAS"):
        fo.fo_adamw_step(bad, torch.bfloat16, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 8)


# ------------------------------------------------------------ full size
def run_full_size(model: W.ModelShape, hyper: W.Hyper, master_bits: int, groups_per_tensor: int = 24,
                  check_steps=(1, 10, 20)):
    rho_bits = 8 if master_bits == 24 else 16
    wid = W.WORKLOAD_IDS[model.name]
    specs = W.llama_tensor_list(model)
    numels = [s.numel for s in specs]
    st = FlashAdamWState(numels, rho_bits=rho_bits, grad_dtype=torch.bfloat16, device=DEV)
    idx, gidx, refs = [], [], []
    for i, s in enumerate(specs):
        gi = W.sample_group_indices(s.numel, groups_per_tensor, seed=1000 + i)
        e = (gi.view(-1, 1) * 32 + torch.arange(32).view(1, -1)).reshape(-1)
        e = e[e < s.numel]
        theta = W.init_theta(s, wid, i, DEV)
        st.init_theta(i, theta)
        refs.append(O.TensorState.init(theta[e.to(DEV)].cpu().numpy(), master_bits=master_bits))
        del theta
        idx.append(e.to(DEV))
        gidx.append(gi.to(DEV))
    for t in range(1, hyper.steps + 1):
        for i, s in enumerate(specs):
            gv = st.grad_view(i)
            W.make_grad(s.numel, wid, i, t, DEV, out=gv)
            gs = gv[idx[i]].cpu().view(torch.int16).numpy().view(np.uint16)
            O.adamw_step(refs[i], gs, t, hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay)
        st.step(t, hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay)
        if t in check_steps:
            torch.cuda.synchronize()
            for i in range(len(specs)):
                v = st.view(i)
                got = {"param": _bits16(v["param"][idx[i]]), "rho": v["rho"][idx[i]].cpu().numpy(),
                       "m": v["m_codes"][idx[i]].cpu().numpy(), "m_scales": _bits16(v["m_scales"][gidx[i]]),
                       "v": v["v_codes"][idx[i]].cpu().numpy(), "v_scales": _bits16(v["v_scales"][gidx[i]])}
                assert_same(got, ref_np(refs[i]), (model.name, specs[i].name, t))
    return st


def test_llama_1b_list_int16_rho_20_steps_sampled():
    st = run_full_size(W.TINYLLAMA_1B, W.TINYLLAMA_HYPER, W.TINYLLAMA_MASTER_BITS)
    assert st.total_numel() == 1_100_048_384 and len(st) == 201


def test_llama3_8b_list_int8_rho_20_steps_sampled():
    st = run_full_size(W.LLAMA3_8B, W.LLAMA3_8B_HYPER, W.LLAMA3_8B_MASTER_BITS, groups_per_tensor=16)
    assert st.total_numel() == 8_030_261_248 and len(st) == 291


@pytest.mark.parametrize("bucket", [0, 5000, 1 << 20])
def test_gradient_release_matches_step(bucket):
    """FlashAdamW(gradient_release=True) steps each parameter inside backward
    and frees its gradient; parameters and states equal those of the normal
    step on the same gradients, bit for bit.  bucket = 0 steps every
    parameter alone, 5000 gathers the biases and the 96 x 48 weight into one
    launch, 2^20 gathers all four."""
    torch.manual_seed(0)

    def model():
        torch.manual_seed(0)
        return torch.nn.Sequential(torch.nn.Linear(64, 96), torch.nn.GELU(), torch.nn.Linear(96, 48)).to(
            device=DEV, dtype=torch.bfloat16)

    a, b = model(), model()
    opt_a = FlashAdamW(a.parameters(), lr=1e-3, weight_decay=0.1)
    opt_b = FlashAdamW(b.parameters(), lr=1e-3, weight_decay=0.1, gradient_release=True,
                       release_bucket_numel=bucket)
    for t in range(3):
        x = torch.randn(32, 64, generator=torch.Generator().manual_seed(t)).to(DEV, torch.bfloat16)
        (a(x).float() ** 2).mean().backward()
        opt_a.step()
        opt_a.zero_grad(set_to_none=True)
        (b(x).float() ** 2).mean().backward()
        assert all(p.grad is None for p in b.parameters())
        opt_b.step()  # nothing left to do
        torch.cuda.synchronize()
        for pa, pb in zip(a.parameters(), b.parameters()):
            assert torch.equal(pa.view(torch.int16), pb.view(torch.int16)), t
            sa, sb = opt_a.state[pa], opt_b.state[pb]
            assert sa["step"] == sb["step"] == t + 1
            for k in ("rho", "m_codes", "m_scales", "v_codes", "v_scales"):
                assert torch.equal(sa[k].view(torch.uint8), sb[k].view(torch.uint8)), (k, t)
    opt_b.remove_hooks()


def test_gradient_release_bucket_left_open_is_stepped_by_step():
    """A small parameter that gets no gradient keeps its bucket from filling:
    the other small parameters keep their gradients through backward and
    step() steps them, equal to the normal step bit for bit."""
    def model():
        torch.manual_seed(1)
        return torch.nn.Sequential(torch.nn.Linear(64, 96), torch.nn.GELU(), torch.nn.Linear(96, 48)).to(
            device=DEV, dtype=torch.bfloat16)

    a, b = model(), model()
    unused = torch.nn.Parameter(torch.zeros(16, dtype=torch.bfloat16, device=DEV))
    opt_a = FlashAdamW(a.parameters(), lr=1e-3, weight_decay=0.1)
    opt_b = FlashAdamW(list(b.parameters()) + [unused], lr=1e-3, weight_decay=0.1, gradient_release=True,
                       release_bucket_numel=5000)
    for t in range(2):
        x = torch.randn(32, 64, generator=torch.Generator().manual_seed(10 + t)).to(DEV, torch.bfloat16)
        (a(x).float() ** 2).mean().backward()
        opt_a.step()
        opt_a.zero_grad(set_to_none=True)
        (b(x).float() ** 2).mean().backward()
        held = [p.grad is not None for p in b.parameters()]
        assert held == [False, True, True, True]  # the 64 x 96 weight alone was released
        opt_b.step()
        assert all(p.grad is None for p in b.parameters()) and unused.grad is None
        torch.cuda.synchronize()
        for pa, pb in zip(a.parameters(), b.parameters()):
            assert torch.equal(pa.view(torch.int16), pb.view(torch.int16)), t
            for k in ("rho", "m_codes", "m_scales", "v_codes", "v_scales"):
                assert torch.equal(opt_a.state[pa][k].view(torch.uint8), opt_b.state[pb][k].view(torch.uint8))
    assert len(opt_b.state[unused]) == 0
    opt_b.remove_hooks()


@pytest.mark.parametrize("bucket", [0, 1 << 20])
def test_gradient_release_matches_oracle(bucket):
    """FlashAdamW(gradient_release=True) steps each parameter from its
    post-accumulate-grad hook and frees the gradient there.  A hook registered
    before the optimizer's captures each gradient as backward completes it;
    the oracle steps the same gradients, and parameters, rho, codes and
    scales must agree bit for bit after every step."""
    net = torch.nn.Sequential(torch.nn.Linear(64, 96), torch.nn.GELU(), torch.nn.Linear(96, 48))
    torch.manual_seed(3)
    net = net.to(device=DEV, dtype=torch.bfloat16)
    params = list(net.parameters())
    refs = [O.TensorState.init(p.detach().float().cpu().numpy().reshape(-1), master_bits=24) for p in params]
    captured = {}
    for i, p in enumerate(params):
        p.register_post_accumulate_grad_hook(lambda q, i=i: captured.__setitem__(i, q.grad.detach().clone()))
    opt = FlashAdamW(params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1, gradient_release=True,
                     release_bucket_numel=bucket)
    for t in range(1, 4):
        captured.clear()
        x = torch.randn(32, 64, generator=torch.Generator().manual_seed(t)).to(DEV, torch.bfloat16)
        (net(x).float() ** 2).mean().backward()
        assert all(p.grad is None for p in params) and len(captured) == len(params)
        for i, p in enumerate(params):
            g = captured[i].reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16)
            O.adamw_step(refs[i], g, t, 1e-3, 0.9, 0.999, 1e-8, 0.1)
        torch.cuda.synchronize()
        for p, r in zip(params, refs):
            s = opt.state[p]
            got = {"param": _bits16(p.detach().reshape(-1)), "rho": s["rho"].cpu().numpy(),
                   "m": s["m_codes"].cpu().numpy(), "m_scales": _bits16(s["m_scales"]),
                   "v": s["v_codes"].cpu().numpy(), "v_scales": _bits16(s["v_scales"])}
            assert_same(got, ref_np(r), ("gradient release", t))
    opt.remove_hooks()


def test_bounded_wait_running_out_is_reported():
    """Failure detection without a fault: a wait that nothing completes gives
    up after its poll limit, the timeout bit reaches the host through
    fo_device_status (which clears it), and the context stays usable."""
    fo.fo_device_status()  # clear anything left by earlier tests
    for polls in (1, 4096):
        fo.fo_check_wait_timeout(polls)
        torch.cuda.synchronize()
        assert fo.fo_device_status() == 1, polls
        assert fo.fo_device_status() == 0
    # the same process goes on stepping bit-exactly
    run_small([4096 + 17, 100], 8, torch.bfloat16, W.LLAMA3_8B_HYPER, 2)
    assert fo.fo_device_status() == 0
    with pytest.raises(fo.FoError):
        fo.fo_check_wait_timeout(0)
