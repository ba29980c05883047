"""Storage bytes per parameter (quantized_state_optimizer_gb300.accounting)
against the page's accounting ("code/flashsim/flash_adamw_sim.py",
`bytes_per_param`, Table 1): its parts for each named configuration, with and
without gradient release, and the slabs a FlashAdamWState actually allocates."""

import pytest
import torch

from quantized_state_optimizer_gb300.accounting import named_bytes_per_param, storage_bytes_per_param
from quantized_state_optimizer_gb300.optim import FlashAdamWState

SCALE = 2 / 32  # the fp16 scale of a group of 32, per element

# the parts the page's accounting lists for each configuration
PAGE = {
    ("adamw_ref", False): {"master": 4, "grad": 4, "m": 4, "v": 4},
    ("flash_adamw", False): {"master": 2, "ecc": 1, "grad": 2, "m": 1 + SCALE, "v": 1 + SCALE},
    ("flash_adamw", True): {"master": 2, "ecc": 1, "grad": 0, "m": 1 + SCALE, "v": 1 + SCALE},
    ("sgd_ref", False): {"master": 4, "grad": 4, "m": 4},
    ("flash_sgd", False): {"master": 2, "ecc": 1, "grad": 2, "m": 1 + SCALE},
    ("flash_sgd", True): {"master": 2, "ecc": 1, "grad": 0, "m": 1 + SCALE},
}


@pytest.mark.parametrize("kind,release", sorted(PAGE))
def test_named_configurations_match_the_page(kind, release):
    got = named_bytes_per_param(kind, gradient_release=release)
    want = PAGE[(kind, release)]
    for part, value in want.items():
        assert got[part] == pytest.approx(value), (kind, part)
    extra = {k: v for k, v in got.items() if k not in want and k != "total"}
    assert all(v == 0 for v in extra.values()), extra
    assert got["total"] == pytest.approx(sum(want.values()))


def test_totals():
    assert named_bytes_per_param("adamw_ref")["total"] == 16
    assert named_bytes_per_param("flash_adamw")["total"] == pytest.approx(7.125)
    assert named_bytes_per_param("flash_adamw", gradient_release=True)["total"] == pytest.approx(5.125)
    assert named_bytes_per_param("sgd_ref")["total"] == 12
    assert named_bytes_per_param("flash_sgd")["total"] == pytest.approx(6.0625)
    assert named_bytes_per_param("flash_sgd", gradient_release=True)["total"] == pytest.approx(4.0625)


def test_ablation_formats_and_errors():
    assert storage_bytes_per_param("bf16_rho16", "linear")["total"] == pytest.approx(2 + 2 + 2 + 2 * (1 + SCALE))
    assert storage_bytes_per_param("bf16", "f32", grad_bytes=4)["total"] == 2 + 4 + 8
    with pytest.raises(ValueError):
        storage_bytes_per_param("fp8", "linear")
    with pytest.raises(ValueError):
        named_bytes_per_param("lion")


def test_flash_adamw_state_allocates_the_accounted_bytes():
    """The slabs of a list whose tensors are multiples of 32 elements hold
    exactly the page's 7.125 B per parameter (bf16 grads, int8 rho)."""
    numels = [4096, 32 * 1000, 1 << 16]
    st = FlashAdamWState(numels, rho_bits=8, grad_dtype=torch.bfloat16, device="cpu")
    assert st.bytes_allocated() / sum(numels) == pytest.approx(named_bytes_per_param("flash_adamw")["total"])
    st16 = FlashAdamWState(numels, rho_bits=16, grad_dtype=torch.bfloat16, device="cpu", with_grads=False)
    assert st16.bytes_allocated() / sum(numels) == pytest.approx(
        storage_bytes_per_param("bf16_rho16", "companded", gradient_release=True)["total"])
