"""ZeRO-style sharding of the FlashAdamW step across data-parallel ranks.

The step updates every group of 32 elements from that group alone: the
group's absmax scales ("code/flashsim/quantization.py", `quantize`) and the
element-wise update of `FlashAdamWSim.step` ("code/flashsim/flash_adamw_sim.py",
Algorithm 4).  So the optimizer state of a list of tensors can be cut at
group boundaries and spread over the ranks of a data-parallel job, each rank
stepping only its own share:

* **Layout.**  The tensors sit in one flat element space, each starting at a
  multiple of ``SHARD_ALIGN`` = 256 elements (8 groups), padded to
  ``world_size`` equal shards whose length is a multiple of 256.  Rank r owns
  the flat range [r C, (r + 1) C).  Its *pieces* are the intersections of that
  range with the tensors: each starts at a multiple of 256 inside its tensor,
  so a piece holds whole groups of the tensor (only a tensor's true end may be
  a ragged group) and every buffer of the piece starts 16-byte aligned, the
  fp16 scale rows included.
* **Buffers.**  theta' (bf16) and the gradient are full-size on every rank
  (the model's parameters and what backward writes).  rho, the momentum and
  variance codes and their scales exist for the rank's shard only.
* **Step.**  ``reduce_grads`` reduce-scatters the gradient (sum) into the
  rank's shard, ``step_shard`` runs ``fo_adamw_step`` over the rank's pieces
  (one launch), and ``sync_params`` all-gathers theta' in place so that every
  rank holds the new parameters.  With one rank no collective runs.

Per parameter and step, a rank moves the fused step's bytes for C elements
and the collectives move the gradient once (reduce-scatter) and theta' once
(all-gather); rho, m and v never leave the rank.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import FoTensor, fo_adamw_step, fo_split, n_groups

SHARD_ALIGN = 256  # elements: 8 groups of 32, so a cut's fp16 scale row starts 16-byte aligned


def _round_up(n: int, k: int) -> int:
    return (n + k - 1) // k * k


@dataclass(frozen=True)
class Piece:
    """The part of one tensor that one rank owns."""

    tensor: int  # index in the list
    start: int   # first element inside the tensor (a multiple of SHARD_ALIGN)
    length: int  # elements
    flat: int    # first element in the flat space

    @property
    def end(self) -> int:
        return self.start + self.length


@dataclass(frozen=True)
class ShardLayout:
    """Flat offsets of a tensor list and its split into equal shards."""

    numels: tuple[int, ...]
    world_size: int
    offsets: tuple[int, ...]  # flat start of each tensor, multiples of SHARD_ALIGN
    shard: int                # elements per rank, a multiple of SHARD_ALIGN

    @property
    def total(self) -> int:
        return self.shard * self.world_size

    def pieces(self, rank: int) -> list[Piece]:
        if not 0 <= rank < self.world_size:
            raise ValueError(f"rank {rank} outside world of {self.world_size}")
        lo, hi = rank * self.shard, (rank + 1) * self.shard
        out = []
        for i, (n, off) in enumerate(zip(self.numels, self.offsets)):
            a, b = max(lo, off), min(hi, off + n)
            if a < b:
                out.append(Piece(i, a - off, b - a, a))
        return out


def shard_layout(numels, world_size: int) -> ShardLayout:
    """Offsets and shard length for ``numels`` over ``world_size`` ranks."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    numels = tuple(int(n) for n in numels)
    if any(n < 0 for n in numels):
        raise ValueError("negative numel")
    offsets, o = [], 0
    for n in numels:
        offsets.append(o)
        o += _round_up(n, SHARD_ALIGN)
    shard = max(_round_up(-(-o // world_size), SHARD_ALIGN), SHARD_ALIGN)
    return ShardLayout(numels, world_size, tuple(offsets), shard)


class ShardedFlashAdamWState:
    """One rank's share of the FlashAdamW state of a tensor list (see the
    module docstring for the layout and the three phases of a step).

    ``rank`` / ``world_size`` default to those of ``process_group`` (or of the
    default group when torch.distributed is initialised, else 0 / 1).  The
    collectives run on ``process_group``; the step itself runs in libfo.so
    and needs CUDA buffers.
    """

    def __init__(self, numels, rho_bits: int = 8, grad_dtype=torch.bfloat16, device="cuda",
                 process_group=None, rank: int | None = None, world_size: int | None = None):
        import torch.distributed as dist
        if rho_bits not in (8, 16):
            raise ValueError("rho_bits must be 8 or 16")
        dist_on = dist.is_available() and dist.is_initialized()
        if world_size is None:
            world_size = dist.get_world_size(process_group) if dist_on else 1
        if rank is None:
            rank = dist.get_rank(process_group) if dist_on else 0
        self.layout = shard_layout(numels, world_size)
        self.rank, self.world_size = rank, world_size
        self.pieces = self.layout.pieces(rank)
        self.rho_bits = rho_bits
        self.grad_dtype = grad_dtype
        self.device = torch.device(device)
        self.process_group = process_group
        L, C = self.layout, self.layout.shard
        dev = self.device
        self.param = torch.zeros(L.total, dtype=torch.bfloat16, device=dev)
        self.grad = torch.zeros(L.total, dtype=grad_dtype, device=dev)
        # with one rank the shard is the whole gradient: no reduce-scatter, no copy
        self.grad_shard = self.grad if world_size == 1 else torch.zeros(C, dtype=grad_dtype, device=dev)
        self.rho = torch.zeros(C, dtype=torch.int8 if rho_bits == 8 else torch.int16, device=dev)
        self.m_codes = torch.zeros(C, dtype=torch.int8, device=dev)
        self.v_codes = torch.zeros(C, dtype=torch.uint8, device=dev)
        self.m_scales = torch.zeros(C // 32, dtype=torch.float16, device=dev)
        self.v_scales = torch.zeros(C // 32, dtype=torch.float16, device=dev)
        self._fo_array = None

    # ------------------------------------------------------------ views
    @property
    def numels(self) -> tuple[int, ...]:
        return self.layout.numels

    @property
    def shard_start(self) -> int:
        return self.rank * self.layout.shard

    def param_view(self, i: int) -> torch.Tensor:
        off = self.layout.offsets[i]
        return self.param[off: off + self.layout.numels[i]]

    def grad_view(self, i: int) -> torch.Tensor:
        off = self.layout.offsets[i]
        return self.grad[off: off + self.layout.numels[i]]

    def piece_views(self, p: Piece) -> dict[str, torch.Tensor]:
        """The buffers of one owned piece (param in the full replica, the rest
        in the shard)."""
        s = p.flat - self.shard_start
        g0, g = s // 32, n_groups(p.length)
        return {"param": self.param[p.flat: p.flat + p.length], "grad": self.grad_shard[s: s + p.length],
                "rho": self.rho[s: s + p.length], "m_codes": self.m_codes[s: s + p.length],
                "v_codes": self.v_codes[s: s + p.length], "m_scales": self.m_scales[g0: g0 + g],
                "v_scales": self.v_scales[g0: g0 + g]}

    # ------------------------------------------------------------ set-up
    def init_theta(self, i: int, theta: torch.Tensor, stream=None) -> None:
        """Split the owned pieces of tensor i's fp32 master weight into theta'
        and rho (``theta`` is the whole tensor; other ranks' parts are not
        read).  ``sync_params`` then gives every rank the whole theta'."""
        flat = theta.reshape(-1)
        for p in self.pieces:
            if p.tensor != i:
                continue
            v = self.piece_views(p)
            fo_split(flat[p.start: p.end].contiguous(), self.rho_bits, v["param"], v["rho"], stream)

    def fo_tensors(self):
        """ctypes ``fo_tensor`` array over the owned pieces (cached)."""
        if self._fo_array is None:
            arr = (FoTensor * max(len(self.pieces), 1))()
            for k, p in enumerate(self.pieces):
                v = self.piece_views(p)
                arr[k] = FoTensor(v["param"].data_ptr(), v["rho"].data_ptr(), v["grad"].data_ptr(),
                                  v["m_codes"].data_ptr(), v["m_scales"].data_ptr(), v["v_codes"].data_ptr(),
                                  v["v_scales"].data_ptr(), p.length)
            self._fo_array = (arr, len(self.pieces))
        return self._fo_array

    # ------------------------------------------------------------ the step
    def reduce_grads(self, op=None) -> None:
        """Sum the ranks' full gradients into this rank's shard
        (reduce-scatter; ``op`` defaults to SUM)."""
        if self.world_size == 1:
            return
        import torch.distributed as dist
        dist.reduce_scatter_tensor(self.grad_shard, self.grad, op=dist.ReduceOp.SUM if op is None else op,
                                   group=self.process_group)

    def step_shard(self, step: int, lr: float, beta1: float, beta2: float, eps: float,
                   weight_decay: float, stream=None) -> None:
        """The fused FlashAdamW step over the owned pieces: one launch."""
        if self.device.type != "cuda":
            raise RuntimeError("the step runs in libfo.so and needs CUDA buffers")
        if not self.pieces:  # a rank whose shard is all padding
            return
        arr, _ = self.fo_tensors()
        fo_adamw_step(arr, self.grad_dtype, lr, beta1, beta2, eps, weight_decay, step, self.rho_bits, stream)

    def sync_params(self) -> None:
        """All-gather theta' in place: every rank gets every shard's new values."""
        if self.world_size == 1:
            return
        import torch.distributed as dist
        C = self.layout.shard
        dist.all_gather_into_tensor(self.param, self.param[self.shard_start: self.shard_start + C],
                                    group=self.process_group)

    def step(self, step: int, lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
             stream=None, op=None) -> None:
        """reduce_grads, step_shard, sync_params."""
        self.reduce_grads(op)
        self.step_shard(step, lr, beta1, beta2, eps, weight_decay, stream)
        self.sync_params()

    # ------------------------------------------------------------ checkpoint
    def state_dict(self) -> dict:
        """Host copies of this rank's shard (and its place in the layout)."""
        return {"rank": self.rank, "world_size": self.world_size, "numels": list(self.layout.numels),
                "rho_bits": self.rho_bits, "param": self.param.cpu(),
                **{k: getattr(self, k).cpu() for k in ("rho", "m_codes", "m_scales", "v_codes", "v_scales")}}

    def load_state_dict(self, sd: dict) -> None:
        if (sd["rank"], sd["world_size"], tuple(sd["numels"]), sd["rho_bits"]) != (
                self.rank, self.world_size, self.layout.numels, self.rho_bits):
            raise ValueError("checkpoint of another rank, world size, tensor list or rho width")
        for k in ("param", "rho", "m_codes", "m_scales", "v_codes", "v_scales"):
            getattr(self, k).copy_(sd[k])


class ZeroFlashAdamW(torch.optim.Optimizer):
    """FlashAdamW over data-parallel ranks with the optimizer state sharded
    (``ShardedFlashAdamWState``).

    The bf16 parameters are re-seated as views of the state's flat theta'
    buffer and their ``.grad`` as views of its flat gradient, so backward
    accumulates straight into the buffer the reduce-scatter reads and the
    all-gather refreshes the parameters the model uses.  ``zero_grad`` zeroes
    that buffer in place (the gradients are never set to None).  Gradients are
    summed over ranks: scale the loss by 1 / world_size for the mean.
    Hyper-parameters come from the first param group; every parameter is
    stepped on every call, as the flat buffers hold them all.
    """

    def __init__(self, params, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 0.01, master_weight_bits: int = 24, process_group=None):
        if master_weight_bits not in (24, 32):
            raise ValueError("master_weight_bits must be 24 or 32")
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay))
        plist = [p for g in self.param_groups for p in g["params"]]
        for p in plist:
            if p.dtype != torch.bfloat16 or not p.is_cuda:
                raise TypeError("ZeroFlashAdamW needs bf16 CUDA parameters")
        self._plist = plist
        self.shard = ShardedFlashAdamWState([p.numel() for p in plist], rho_bits=8 if master_weight_bits == 24 else 16,
                                            grad_dtype=torch.bfloat16, device=plist[0].device,
                                            process_group=process_group)
        with torch.no_grad():
            for i, p in enumerate(plist):
                self.shard.init_theta(i, p.detach().float())
            self.shard.sync_params()
            for i, p in enumerate(plist):
                p.data = self.shard.param_view(i).view_as(p)
                p.grad = self.shard.grad_view(i).view_as(p)
        self._t = 0

    def zero_grad(self, set_to_none: bool = False) -> None:
        self.shard.grad.zero_()

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        g = self.param_groups[0]
        self._t += 1
        b1, b2 = g["betas"]
        self.shard.step(self._t, g["lr"], b1, b2, g["eps"], g["weight_decay"])
        return loss
