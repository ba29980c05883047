"""Pins of the oracle's number-format conversions against torch's own conversions.

The quantization page stores group scales with ``Tensor.to(torch.float16)``
and the harness page rounds parameters with ``Tensor.to(torch.bfloat16)``;
the oracle re-implements both on bit patterns, so here they are checked
against the library routines they stand for.
"""

import numpy as np
import torch

import oracle as O


def _all_exponent_sweep(per_exp=2048, seed=3):
    rng = np.random.default_rng(seed)
    exps = np.repeat(np.arange(256, dtype=np.uint32), per_exp)
    mant = rng.integers(0, 1 << 23, exps.size, dtype=np.uint32)
    sign = rng.integers(0, 2, exps.size, dtype=np.uint32) << 31
    bits = sign | (exps << 23) | mant
    # boundaries of the half range and exact ties
    extra = np.array([0x00000000, 0x80000000, 0x477FE000, 0x477FEFFF, 0x477FF000, 0x477FF001,
                      0x47800000, 0x33800000, 0x33000000, 0x33000001, 0x387FC000, 0x38800000,
                      0x7F800000, 0xFF800000, 0x3F801000, 0x3F803000, 0x3F800FFF, 0x3F801001],
                     dtype=np.uint32)
    return np.concatenate([bits, extra]).view(np.float32)


def test_f32_to_f16_matches_torch():
    x = _all_exponent_sweep()
    ours = O.f32_to_f16_bits(x)
    ref = torch.from_numpy(x.copy()).half().view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (payload is not part of the method)
    oh = ours[nan]
    assert np.all(((oh >> 10) & 0x1F) == 0x1F) and np.all((oh & 0x3FF) != 0)


def test_f32_to_f16_dense_near_half_range():
    # every 31st fp32 pattern in [2^-26, 2^17): all binades, subnormal and overflow edges
    lo, hi = 0x32800000, 0x48000000
    bits = np.arange(lo, hi, 31, dtype=np.uint32)
    x = bits.view(np.float32)
    ours = O.f32_to_f16_bits(x)
    ref = torch.from_numpy(x.copy()).half().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_to_f32_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_bits_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.float16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_bf16_rne_matches_torch():
    x = _all_exponent_sweep(seed=5)
    ours = O.f32_to_bf16_rne_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # explicit ties both ways
    t = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x7F7F8000], dtype=np.uint32).view(np.float32)
    ref_t = torch.from_numpy(t.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_rne_bits(t), ref_t)
