"""Seeded synthetic inputs for the fused FlashAdamW step and its kernel pairs.

This module only *draws* inputs: it holds none of the method's arithmetic
(no quantization, no splitting, no optimizer update).  Both the CPU oracle
(tests only) and the CUDA path take their inputs from here, so that the two
sides see identical bytes without either one importing the other.

Workloads (the pages measure on no public dataset; everything is synthetic):

* ``battery()`` -- the seven test tensors of the equivalence harness page
  (code/gpu/equivalence.py, ``battery``): a CPU generator seeded with 7, drawn
  in the listed order (for ``heavy_tail`` the outer ``randn`` before the one
  inside ``exp``; for ``with_zeros`` the ``rand`` mask before the ``randn``).
* ``exponent_sweep()`` -- the stratified fp32 sweep of the same page
  (``eq_ecc``): exponents 1, 5, ..., 253, 2^16 uniform 23-bit mantissas per
  exponent, global torch seed 11, optional random sign.
* ``single_tensor_theta()/single_tensor_grad()`` -- one flat tensor of
  2^16+17 parameters, theta ~ N(0, 0.02) (seed 0), grads ~ N(0, 1e-3) with
  seed 1000+t at step t.
* ``llama_tensor_list()`` -- the parameter shapes of a 1.1B TinyLlama-like
  model (hidden 2048, ffn 5632, 22 layers, 32 query / 4 KV heads of 64,
  vocab 32000, untied head) and of Llama-3-8B (hidden 4096, ffn 14336,
  32 layers, 32 query / 8 KV heads of 128, vocab 128256, untied head).
  Matrices start at theta ~ N(0, 0.02), norm weights at 1.0; bf16 grads are
  the round-to-nearest-even bf16 of N(0, 1e-3), drawn per (tensor, step)
  from a seed that mixes the workload id, the tensor index and the step.
"""

from __future__ import annotations

import dataclasses

import torch

GROUP = 32


# --------------------------------------------------------------------------
# Quantize / dequantize battery (equivalence harness page, ``battery``)
# --------------------------------------------------------------------------
def battery() -> dict[str, torch.Tensor]:
    """The seven fp32 CPU tensors of the harness, seed 7, in draw order."""
    g = torch.Generator(device="cpu").manual_seed(7)
    ts = {}
    ts["normal"] = torch.randn(1 << 20, generator=g)
    outer = torch.randn(1 << 20, generator=g)
    inner = torch.randn(1 << 20, generator=g)
    ts["heavy_tail"] = outer * torch.exp(inner * 3)
    ts["tiny"] = torch.randn(1 << 16, generator=g) * 1e-20
    ts["adam_v_like"] = (torch.randn(1 << 20, generator=g) * 1e-3) ** 2
    ts["nonmult32"] = torch.randn((1 << 16) + 17, generator=g)
    ts["const_groups"] = torch.ones(1 << 12) * 0.37
    mask = torch.rand(1 << 16, generator=g) < 0.3
    vals = torch.randn(1 << 16, generator=g)
    ts["with_zeros"] = torch.where(mask, torch.zeros(1), vals)
    return ts


# --------------------------------------------------------------------------
# Split / reconstruct exponent sweep (equivalence harness page, ``eq_ecc``)
# --------------------------------------------------------------------------
SWEEP_EXPONENTS = list(range(1, 255, 4))
SWEEP_PER_EXPONENT = 1 << 16


def exponent_sweep(random_sign: bool = True, per_exp: int = SWEEP_PER_EXPONENT) -> torch.Tensor:
    """fp32 values with uniform 23-bit mantissas in each exponent bucket.

    Returns a 1-D fp32 CPU tensor of ``len(SWEEP_EXPONENTS) * per_exp`` values.
    The global torch RNG is seeded with 11 as on the page; it is saved and
    restored around the draw so that callers' RNG state is untouched.
    """
    state = torch.random.get_rng_state()
    try:
        torch.manual_seed(11)
        chunks = []
        for e in SWEEP_EXPONENTS:
            mant = torch.randint(0, 1 << 23, (per_exp,), dtype=torch.int32)
            bits = (e << 23) | mant
            if random_sign:
                sign = torch.randint(0, 2, (per_exp,), dtype=torch.int32) << 31
                bits = sign | bits
            chunks.append(bits.view(torch.float32))
        return torch.cat(chunks)
    finally:
        torch.random.set_rng_state(state)


# --------------------------------------------------------------------------
# Single flat tensor (2^16 + 17 parameters, fp32 grads)
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Hyper:
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    steps: int


SINGLE_TENSOR_NUMEL = (1 << 16) + 17
SINGLE_TENSOR_HYPER = Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, steps=10)


def single_tensor_theta(numel: int = SINGLE_TENSOR_NUMEL) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(0)
    return torch.randn(numel, generator=g) * 0.02


def single_tensor_grad(step: int, numel: int = SINGLE_TENSOR_NUMEL) -> torch.Tensor:
    """fp32 grad for step ``step`` (1-based), seed 1000 + step."""
    g = torch.Generator(device="cpu").manual_seed(1000 + step)
    return torch.randn(numel, generator=g) * 1e-3


# --------------------------------------------------------------------------
# Llama-shaped tensor lists
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    vocab: int
    hidden: int
    ffn: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int


TINYLLAMA_1B = ModelShape("llama-1.1b", vocab=32000, hidden=2048, ffn=5632, layers=22,
                          q_heads=32, kv_heads=4, head_dim=64)
LLAMA3_8B = ModelShape("llama-3-8b", vocab=128256, hidden=4096, ffn=14336, layers=32,
                       q_heads=32, kv_heads=8, head_dim=128)

# Hyper-parameters of the two multi-tensor workloads.  For the 1.1B list only
# wd = 0.1 and 20 steps are given; lr / betas / eps are taken from the single
# tensor case.
TINYLLAMA_HYPER = Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, steps=20)
LLAMA3_8B_HYPER = Hyper(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, steps=20)

# master weight width of each multi-tensor workload: 32-bit (int16 rho) for the
# 1.1B list, 24-bit (int8 rho) for the 8B list
TINYLLAMA_MASTER_BITS = 32
LLAMA3_8B_MASTER_BITS = 24


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple[int, ...]
    is_norm: bool

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def llama_tensor_list(m: ModelShape) -> list[TensorSpec]:
    """Parameter tensors of a Llama-style decoder in module order."""
    h, kv = m.hidden, m.kv_heads * m.head_dim
    out = [TensorSpec("embed_tokens", (m.vocab, h), False)]
    for i in range(m.layers):
        p = f"layers.{i}."
        out += [
            TensorSpec(p + "input_layernorm", (h,), True),
            TensorSpec(p + "q_proj", (m.q_heads * m.head_dim, h), False),
            TensorSpec(p + "k_proj", (kv, h), False),
            TensorSpec(p + "v_proj", (kv, h), False),
            TensorSpec(p + "o_proj", (h, m.q_heads * m.head_dim), False),
            TensorSpec(p + "post_attention_layernorm", (h,), True),
            TensorSpec(p + "gate_proj", (m.ffn, h), False),
            TensorSpec(p + "up_proj", (m.ffn, h), False),
            TensorSpec(p + "down_proj", (h, m.ffn), False),
        ]
    out.append(TensorSpec("norm", (h,), True))
    out.append(TensorSpec("lm_head", (m.vocab, h), False))
    return out


WORKLOAD_IDS = {"llama-1.1b": 4, "llama-3-8b": 5}


def _mix(*xs: int) -> int:
    """64-bit integer mix of a few small ints (splitmix64 finaliser) -> 63-bit seed."""
    z = 0x9E3779B97F4A7C15
    for x in xs:
        z = (z + (x & 0xFFFFFFFFFFFFFFFF) + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        z ^= z >> 31
    return z & 0x7FFFFFFFFFFFFFFF


def theta_seed(workload_id: int, tensor_idx: int) -> int:
    return _mix(workload_id, tensor_idx, 0xA11CE)


def grad_seed(workload_id: int, tensor_idx: int, step: int) -> int:
    return _mix(workload_id, tensor_idx, step)


def init_theta(spec: TensorSpec, workload_id: int, tensor_idx: int, device) -> torch.Tensor:
    """fp32 initial master weight of one tensor (flat)."""
    if spec.is_norm:
        return torch.ones(spec.numel, dtype=torch.float32, device=device)
    g = torch.Generator(device=device).manual_seed(theta_seed(workload_id, tensor_idx))
    t = torch.randn(spec.numel, generator=g, device=device, dtype=torch.float32)
    return t.mul_(0.02)


def make_grad(numel: int, workload_id: int, tensor_idx: int, step: int, device,
              dtype=torch.bfloat16, out: torch.Tensor | None = None) -> torch.Tensor:
    """Grad of one tensor at one step: dtype(N(0, 1e-3)), flat."""
    g = torch.Generator(device=device).manual_seed(grad_seed(workload_id, tensor_idx, step))
    t = torch.randn(numel, generator=g, device=device, dtype=torch.float32).mul_(1e-3)
    if out is None:
        return t.to(dtype)
    out.copy_(t)
    return out


def sample_group_indices(numel: int, k: int, seed: int) -> torch.Tensor:
    """``k`` distinct group indices of a tensor (sorted), always including its last group."""
    n_groups = (numel + GROUP - 1) // GROUP
    if k >= n_groups:
        return torch.arange(n_groups, dtype=torch.int64)
    g = torch.Generator(device="cpu").manual_seed(seed)
    idx = torch.randperm(n_groups - 1, generator=g)[: k - 1]
    idx = torch.cat([idx, torch.tensor([n_groups - 1])])
    return torch.sort(idx).values
