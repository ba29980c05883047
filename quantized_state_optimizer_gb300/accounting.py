"""Storage bytes per parameter of an optimizer's state in HBM.

The accounting the paper tabulates ("code/flashsim/flash_adamw_sim.py",
`bytes_per_param`, Table 1): what one parameter costs in memory between
steps -- the master weight (or theta' and its residual rho), the gradient
buffer (none when the step runs inside backward, "gradient release"), and
each optimizer state, a quantized state costing one code byte plus its share
of the fp16 scale of its group of 32.

Here the totals are derived from the storage formats themselves, so that the
same function covers the formats of ``fo_adamw_step_general`` and
``fo_sgd_step``; tests/test_accounting_cpu.py checks the paper's totals.
"""

from __future__ import annotations

GROUP = 32
SCALE_BYTES = 2  # one fp16 scale per group

_PARAM_BYTES = {  # bytes of the parameter and of its residual, by format
    "f32": (4, 0),
    "bf16": (2, 0),
    "bf16_rho8": (2, 1),
    "bf16_rho16": (2, 2),
}


def state_bytes(state_format: str) -> float:
    """One optimizer state per parameter: a code byte plus 2/32 of an fp16
    scale (companded or linear codes), or an fp32 value."""
    if state_format in ("companded", "linear"):
        return 1 + SCALE_BYTES / GROUP
    if state_format == "f32":
        return 4.0
    raise ValueError(f"state format {state_format!r}")


def storage_bytes_per_param(param_format: str, state_format: str, optimizer: str = "adamw",
                            grad_bytes: int = 2, gradient_release: bool = False) -> dict[str, float]:
    """Per-parameter storage, by component and in total.

    ``optimizer`` "adamw" keeps two states (m, v), "sgd" one (the momentum
    buffer).  ``grad_bytes`` is the width of the gradient buffer (2 for bf16,
    4 for fp32); with ``gradient_release`` no gradient buffer persists.
    """
    if param_format not in _PARAM_BYTES:
        raise ValueError(f"parameter format {param_format!r}")
    if optimizer not in ("adamw", "sgd"):
        raise ValueError(f"optimizer {optimizer!r}")
    param, rho = _PARAM_BYTES[param_format]
    parts = {"master": float(param), "ecc": float(rho), "grad": 0.0 if gradient_release else float(grad_bytes)}
    parts["m"] = state_bytes(state_format)
    if optimizer == "adamw":
        parts["v"] = state_bytes(state_format)
    parts["total"] = sum(parts.values())
    return parts


# The paper's named configurations (Table 1), as storage formats.
NAMED = {
    "adamw_ref": dict(param_format="f32", state_format="f32", optimizer="adamw", grad_bytes=4),
    "flash_adamw": dict(param_format="bf16_rho8", state_format="companded", optimizer="adamw", grad_bytes=2),
    "sgd_ref": dict(param_format="f32", state_format="f32", optimizer="sgd", grad_bytes=4),
    "flash_sgd": dict(param_format="bf16_rho8", state_format="companded", optimizer="sgd", grad_bytes=2),
}


def named_bytes_per_param(kind: str, gradient_release: bool = False) -> dict[str, float]:
    """Storage of one of the paper's named configurations."""
    if kind not in NAMED:
        raise ValueError(f"unknown configuration {kind!r}")
    return storage_bytes_per_param(**NAMED[kind], gradient_release=gradient_release)
