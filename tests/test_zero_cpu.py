"""ZeRO-style sharding (quantized_state_optimizer_gb300.zero) on the CPU.

* The layout: every element of every tensor belongs to exactly one rank,
  pieces start on 256-element boundaries (whole groups, 16-byte-aligned scale
  rows) and stay inside their rank's shard.
* Two gloo ranks run the real reduce-scatter and all-gather around the
  rank-local step.  The test swaps the kernel launch for the oracle (a
  subclass that overrides ``init_theta`` / ``step_shard``; the library itself
  has no CPU step), and both ranks must end with the state a single process
  gets by stepping every tensor with the summed gradient.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from quantized_state_optimizer_gb300.zero import SHARD_ALIGN, ShardedFlashAdamWState, shard_layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUMELS = [70000, 4097, 33, 0, 1, 100003, 256 * 5, 31]
H = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05)


@pytest.mark.parametrize("ws", [1, 2, 3, 4, 7, 8])
def test_layout_covers_every_element_once(ws):
    rng = np.random.default_rng(ws)
    for numels in (NUMELS, [int(x) for x in rng.integers(0, 5000, 40)], [3], [0, 0]):
        L = shard_layout(numels, ws)
        assert L.shard % SHARD_ALIGN == 0 and L.total == L.shard * ws
        assert all(o % SHARD_ALIGN == 0 for o in L.offsets)
        assert L.total >= L.offsets[-1] + numels[-1]
        owner = [np.full(n, -1) for n in numels]
        for r in range(ws):
            lo, hi = r * L.shard, (r + 1) * L.shard
            for p in L.pieces(r):
                assert p.start % SHARD_ALIGN == 0 and p.flat % SHARD_ALIGN == 0
                assert (p.flat - lo) % SHARD_ALIGN == 0
                assert lo <= p.flat and p.flat + p.length <= hi
                assert p.flat == L.offsets[p.tensor] + p.start and p.length > 0
                assert (owner[p.tensor][p.start: p.end] == -1).all()
                owner[p.tensor][p.start: p.end] = r
        assert all((o >= 0).all() for o in owner)


def test_layout_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard_layout([4], 0)
    with pytest.raises(ValueError):
        shard_layout([-1], 2)
    with pytest.raises(ValueError):
        shard_layout([4], 2).pieces(2)


def test_step_needs_cuda_buffers():
    st = ShardedFlashAdamWState([100], device="cpu", rank=0, world_size=1)
    with pytest.raises(RuntimeError):
        st.step_shard(1, **H)


def test_checkpoint_of_another_rank_is_refused():
    a = ShardedFlashAdamWState(NUMELS, device="cpu", rank=0, world_size=2)
    b = ShardedFlashAdamWState(NUMELS, device="cpu", rank=1, world_size=2)
    a.m_codes.fill_(3)
    sd = a.state_dict()
    with pytest.raises(ValueError):
        b.load_state_dict(sd)
    c = ShardedFlashAdamWState(NUMELS, device="cpu", rank=0, world_size=2)
    c.load_state_dict(sd)
    assert torch.equal(c.m_codes, a.m_codes)


# ------------------------------------------------------------ two gloo ranks
def _u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


class OracleShard(ShardedFlashAdamWState):
    """The rank-local work done by the oracle instead of libfo.so (CPU test)."""

    def init_theta(self, i, theta, stream=None):
        mb = 24 if self.rho_bits == 8 else 32
        for p in self.pieces:
            if p.tensor != i:
                continue
            hi, rho = O.split(theta.reshape(-1)[p.start: p.end].numpy(), mb)
            v = self.piece_views(p)
            v["param"].view(torch.int16).copy_(torch.from_numpy(hi.view(np.int16)))
            v["rho"].copy_(torch.from_numpy(rho))

    def step_shard(self, step, lr, beta1, beta2, eps, weight_decay, stream=None):
        kind = O.PARAM_BF16_RHO8 if self.rho_bits == 8 else O.PARAM_BF16_RHO16
        for p in self.pieces:
            v = self.piece_views(p)
            st = O.TensorState(_u16(v["param"]), v["rho"].numpy(), v["m_codes"].numpy(), _u16(v["m_scales"]),
                               v["v_codes"].numpy(), _u16(v["v_scales"]), kind)
            O.adamw_step(st, v["grad"].numpy(), step, lr, beta1, beta2, eps, weight_decay)


def _theta(i, n):
    g = torch.Generator().manual_seed(900 + i)
    return torch.randn(n, generator=g) * 0.02


def _grad(rank, i, t, n):
    """Multiples of 2^-20 below 2^-7 in magnitude: sums over a few ranks are
    exact in fp32, whatever order the reduction takes."""
    g = torch.Generator().manual_seed(10000 * rank + 100 * i + t)
    return torch.round(torch.randn(n, generator=g) * 1e-3 * 2.0 ** 20).clamp(-8000, 8000) * 2.0 ** -20


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rho_bits, steps, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        st = OracleShard(NUMELS, rho_bits=rho_bits, grad_dtype=torch.float32, device="cpu")
        assert (st.rank, st.world_size) == (rank, world)
        for i, n in enumerate(NUMELS):
            st.init_theta(i, _theta(i, n))
        st.sync_params()
        for t in range(1, steps + 1):
            st.grad.zero_()
            for i, n in enumerate(NUMELS):
                st.grad_view(i).copy_(_grad(rank, i, t, n))
            st.step(t, **H)
        res = {"param": [_u16(st.param_view(i)).copy() for i in range(len(NUMELS))], "pieces": []}
        for p in st.pieces:
            v = st.piece_views(p)
            res["pieces"].append((p.tensor, p.start, p.length, v["rho"].numpy().copy(), v["m_codes"].numpy().copy(),
                                  _u16(v["m_scales"]).copy(), v["v_codes"].numpy().copy(),
                                  _u16(v["v_scales"]).copy()))
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,rho_bits", [(2, 8), (3, 16)])
def test_gloo_ranks_match_one_process(world, rho_bits):
    steps = 3
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), rho_bits, steps, out), nprocs=world,
                       start_method="spawn", join=True)
    # one process: every tensor stepped whole with the summed gradient
    refs = [O.TensorState.init(_theta(i, n).numpy(), master_bits=24 if rho_bits == 8 else 32)
            for i, n in enumerate(NUMELS)]
    for t in range(1, steps + 1):
        for i, n in enumerate(NUMELS):
            if n == 0:
                continue
            g = np.zeros(n, np.float32)
            for r in range(world):
                g = g + _grad(r, i, t, n).numpy()  # exact in any order
            O.adamw_step(refs[i], g, t, **H)
    covered = [0] * len(NUMELS)
    for r in range(world):
        res = out[r]
        for i, ref in enumerate(refs):
            assert np.array_equal(res["param"][i], ref.param), (r, i)
        for (i, start, length, rho, m, ms, v, vs) in res["pieces"]:
            g0, g = start // 32, (length + 31) // 32
            ref = refs[i]
            assert np.array_equal(rho, ref.rho[start: start + length]), (r, i)
            assert np.array_equal(m, ref.m[start: start + length]), (r, i)
            assert np.array_equal(v, ref.v[start: start + length]), (r, i)
            assert np.array_equal(ms, ref.m_scales[g0: g0 + g]), (r, i)
            assert np.array_equal(vs, ref.v_scales[g0: g0 + g]), (r, i)
            covered[i] += length
    assert covered == NUMELS
