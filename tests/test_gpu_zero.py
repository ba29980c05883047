"""ZeRO-style sharding with the real kernel on one GPU.

The ranks of a 2- or 3-rank job are emulated in one process: each rank's
``ShardedFlashAdamWState`` gets its shard of the summed gradient and runs
``step_shard`` (the fused kernel over its pieces); the all-gather is emulated
by copying each rank's shard of theta' into the others.  Every tensor must
come out bit for bit as the unsharded ``FlashAdamWState`` step leaves it, and
each rank's shard of rho, codes and scales must equal the same elements of
the unsharded state.  The collectives themselves are covered on gloo ranks
(tests/test_zero_cpu.py)."""

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from quantized_state_optimizer_gb300.optim import FlashAdamW, FlashAdamWState
from quantized_state_optimizer_gb300.zero import ShardedFlashAdamWState, ZeroFlashAdamW

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
NUMELS = [70000, 4097, 33, 0, 7680 * 3, 1, 100003, 256 * 5]


def _theta(i, n):
    g = torch.Generator().manual_seed(40 + i)
    return torch.randn(n, generator=g) * 0.02


def _grad(i, t, n):
    g = torch.Generator().manual_seed(W.grad_seed(31, i, t))
    return (torch.randn(n, generator=g) * 1e-3).to(torch.bfloat16)


def _gather(shards):
    C = shards[0].layout.shard
    for r, src in enumerate(shards):
        part = src.param[r * C: (r + 1) * C]
        for dst in shards:
            if dst is not src:
                dst.param[r * C: (r + 1) * C].copy_(part)


def _eq(a, b, ctx):
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), ctx


@pytest.mark.parametrize("ws", [2, 3])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_shards_equal_the_unsharded_step(ws, rho_bits):
    h = W.LLAMA3_8B_HYPER
    ref = FlashAdamWState(NUMELS, rho_bits=rho_bits, grad_dtype=torch.bfloat16, device=DEV)
    shards = [ShardedFlashAdamWState(NUMELS, rho_bits=rho_bits, device=DEV, rank=r, world_size=ws)
              for r in range(ws)]
    for i, n in enumerate(NUMELS):
        th = _theta(i, n).to(DEV)
        if n:
            ref.init_theta(i, th)
        for sh in shards:
            sh.init_theta(i, th)
    _gather(shards)
    C = shards[0].layout.shard
    for t in (1, 2, 3):
        flat = torch.zeros(shards[0].layout.total, dtype=torch.bfloat16, device=DEV)
        for i, n in enumerate(NUMELS):
            g = _grad(i, t, n).to(DEV)
            ref.grad_view(i).copy_(g)
            off = shards[0].layout.offsets[i]
            flat[off: off + n].copy_(g)
        ref.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        for r, sh in enumerate(shards):
            sh.grad_shard.copy_(flat[r * C: (r + 1) * C])
            sh.step_shard(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        _gather(shards)
        torch.cuda.synchronize()
        for i, n in enumerate(NUMELS):
            for sh in shards:
                _eq(sh.param_view(i), ref.view(i)["param"], (ws, rho_bits, t, i, "param"))
        for sh in shards:
            for p in sh.pieces:
                v, rv = sh.piece_views(p), ref.view(p.tensor)
                g0, g = p.start // 32, (p.length + 31) // 32
                ctx = (ws, rho_bits, t, sh.rank, p)
                _eq(v["rho"], rv["rho"][p.start: p.end], ctx)
                _eq(v["m_codes"], rv["m_codes"][p.start: p.end], ctx)
                _eq(v["v_codes"], rv["v_codes"][p.start: p.end], ctx)
                _eq(v["m_scales"], rv["m_scales"][g0: g0 + g], ctx)
                _eq(v["v_scales"], rv["v_scales"][g0: g0 + g], ctx)


def _bits(t):
    return t.cpu().view(torch.uint8).numpy()


@pytest.mark.parametrize("ws", [2, 3])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_shards_match_the_oracle_on_summed_gradients(ws, rho_bits):
    """Each emulated rank holds its own gradients; their sum (what the
    reduce-scatter delivers: fp32 sum over ranks, rounded to bf16) reaches each
    rank as its shard, and the rank steps its pieces with the fused kernel.
    The oracle steps whole tensors with the same summed gradient; every rank's
    pieces of rho, codes and scales, and the gathered theta', must equal the
    oracle's elements bit for bit."""
    h = W.LLAMA3_8B_HYPER
    master = 24 if rho_bits == 8 else 32
    shards = [ShardedFlashAdamWState(NUMELS, rho_bits=rho_bits, device=DEV, rank=r, world_size=ws)
              for r in range(ws)]
    refs = []
    for i, n in enumerate(NUMELS):
        th = _theta(i, n)
        refs.append(O.TensorState.init(th.numpy(), master_bits=master))
        for sh in shards:
            sh.init_theta(i, th.to(DEV))
    _gather(shards)
    C = shards[0].layout.shard
    for t in (1, 2, 3):
        flat = torch.zeros(shards[0].layout.total, dtype=torch.bfloat16, device=DEV)
        for i, n in enumerate(NUMELS):
            local = [_grad(i + 1000 * r, t, n).float() for r in range(ws)]
            g = torch.stack(local).sum(0).to(torch.bfloat16)
            off = shards[0].layout.offsets[i]
            flat[off: off + n].copy_(g.to(DEV))
            O.adamw_step(refs[i], g.view(torch.int16).numpy().view(np.uint16), t, h.lr, h.beta1, h.beta2, h.eps,
                         h.weight_decay)
        for r, sh in enumerate(shards):
            sh.grad_shard.copy_(flat[r * C: (r + 1) * C])
            sh.step_shard(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)
        _gather(shards)
        torch.cuda.synchronize()
        for i, n in enumerate(NUMELS):
            for sh in shards:
                got = sh.param_view(i).cpu().view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(got, refs[i].param), (ws, rho_bits, t, i, "param")
        for sh in shards:
            for p in sh.pieces:
                v, r = sh.piece_views(p), refs[p.tensor]
                g0, g = p.start // 32, (p.length + 31) // 32
                ctx = (ws, rho_bits, t, sh.rank, p)
                assert np.array_equal(_bits(v["rho"]), r.rho[p.start: p.end].view(np.uint8)), ctx
                assert np.array_equal(_bits(v["m_codes"]), r.m[p.start: p.end].view(np.uint8)), ctx
                assert np.array_equal(_bits(v["v_codes"]), r.v[p.start: p.end].view(np.uint8)), ctx
                assert np.array_equal(_bits(v["m_scales"]), r.m_scales[g0: g0 + g].view(np.uint8)), ctx
                assert np.array_equal(_bits(v["v_scales"]), r.v_scales[g0: g0 + g].view(np.uint8)), ctx


def test_zero_optimizer_single_rank_matches_flash_adamw():
    torch.manual_seed(0)
    shapes = [(64, 33), (4097,), (7,), (300, 40)]
    init = [(torch.randn(s) * 0.02).to(torch.bfloat16) for s in shapes]
    a = [torch.nn.Parameter(x.clone().to(DEV)) for x in init]
    b = [torch.nn.Parameter(x.clone().to(DEV)) for x in init]
    opt_a = FlashAdamW(a, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    opt_b = ZeroFlashAdamW(b, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    assert opt_b.shard.world_size == 1
    for t in range(1, 4):
        opt_b.zero_grad()
        for i, (pa, pb) in enumerate(zip(a, b)):
            g = _grad(i, t, pa.numel()).reshape(pa.shape).to(DEV)
            pa.grad = g.clone()
            pb.grad.add_(g)  # what backward's accumulation does to the flat view
        opt_a.step()
        opt_b.step()
        torch.cuda.synchronize()
        for pa, pb in zip(a, b):
            _eq(pa.detach(), pb.detach(), t)
    for i, pa in enumerate(a):
        s = opt_a.state[pa]
        v = opt_b.shard.piece_views(opt_b.shard.pieces[i])
        _eq(s["rho"].reshape(-1), v["rho"], i)
        _eq(s["m_codes"].reshape(-1), v["m_codes"], i)
        _eq(s["v_codes"].reshape(-1), v["v_codes"], i)


def test_zero_optimizer_backward_writes_the_flat_gradient():
    """A model whose parameters the optimizer re-seated: backward accumulates
    into the flat gradient buffer and the step changes the model's weights."""
    torch.manual_seed(1)
    net = torch.nn.Sequential(torch.nn.Linear(32, 64), torch.nn.Tanh(), torch.nn.Linear(64, 8)).to(
        device=DEV, dtype=torch.bfloat16)
    opt = ZeroFlashAdamW(net.parameters(), lr=1e-2)
    before = [p.detach().clone() for p in net.parameters()]
    x = torch.randn(16, 32, device=DEV, dtype=torch.bfloat16)
    opt.zero_grad()
    (net(x).float() ** 2).mean().backward()
    assert float(opt.shard.grad.float().abs().sum()) > 0
    for i, p in enumerate(net.parameters()):
        assert p.grad.data_ptr() == opt.shard.grad_view(i).data_ptr()
    opt.step()
    torch.cuda.synchronize()
    assert any(not torch.equal(b, p.detach()) for b, p in zip(before, net.parameters()))
    assert all(np.isfinite(p.detach().float().cpu().numpy()).all() for p in net.parameters())
