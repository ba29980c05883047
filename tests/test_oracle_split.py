"""Pins of the oracle's split / reconstruct (the compute_ecc_bits /
reconstruct_fp32_param pair of the harness page "code/gpu/equivalence.py",
``eq_ecc``, with a 3- or 4-byte master weight).

The pages do not print the pair's source; the reading under test is: the
master is theta rounded to an M-bit float (nearest, ties away from zero),
theta' is the master rounded to bf16 the same way, rho is the exact residual.
These tests pin that reading to things other than the oracle: all 2^32
inputs for the 32-bit master, an independent binary64 rounding of the 24-bit
master, and torch's bf16 rounding away from exact ties.
"""

import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


from _split_ranges import round_to_master24_f64  # noqa: E402
import _split_ranges as R  # noqa: E402


def _over_all_patterns(fn, parts: int = 16):
    """fn over 2^32 bit patterns cut into `parts` ranges, on a spawned pool
    (every range is independent); the failures found."""
    import multiprocessing as mp
    edges = [((1 << 32) * k) // parts for k in range(parts + 1)]
    # ranges start on multiples of 97 so the stride sample is the same as one pass
    edges = [e - e % 97 if 0 < e < (1 << 32) else e for e in edges] if fn is R._master24_stride_range else edges
    workers = max(1, min(parts, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        out = pool.starmap(fn, [(edges[k], edges[k + 1]) for k in range(parts)])
    return [r for r in out if r is not None]


@pytest.mark.slow
def test_master32_round_trip_exhaustive():
    """Every one of the 2^32 fp32 bit patterns reconstructs bit for bit
    (NaNs reconstruct as NaN)."""
    assert _over_all_patterns(R._round_trip32_range) == []


@pytest.mark.slow
def test_master24_matches_binary64_rounding_exhaustive_stride():
    assert _over_all_patterns(R._master24_stride_range) == []


def test_master24_on_sweep_and_bound():
    x = W.exponent_sweep(random_sign=True).numpy()
    hi, rho = O.split(x, 24)
    assert rho.dtype == np.int8
    back = O.reconstruct(hi, rho, 24)
    assert np.array_equal(back.astype(np.float64), round_to_master24_f64(x))
    rel = np.abs(back.astype(np.float64) - x) / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -16
    # the whole int8 range is used
    assert rho.min() == -128 and rho.max() == 127


def test_master32_on_sweep_exact():
    for sign in (False, True):
        x = W.exponent_sweep(random_sign=sign).numpy()
        hi, rho = O.split(x, 32)
        assert rho.dtype == np.int16
        assert np.array_equal(O.reconstruct(hi, rho, 32).view(np.uint32), x.view(np.uint32))


def test_theta_prime_is_torch_bf16_except_ties():
    rng = np.random.default_rng(23)
    bits = rng.integers(0, 1 << 32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, (bits & 0xFFFF0000) | 0x8000])  # add exact ties
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    hi32, _ = O.split(x, 32)
    tie = (x.view(np.uint32) & 0xFFFF) == 0x8000
    assert tie.sum() > 1000
    assert np.array_equal(hi32[~tie], ref[~tie])
    # at a tie theta' is the neighbour away from zero: the magnitude rounds up
    up = (((x[tie].view(np.uint32) >> 16) + 1) & 0x7FFF).astype(np.uint16)
    assert np.array_equal(hi32[tie] & 0x7FFF, up)
    # 24-bit master: theta' is the bf16 rounding of the master itself
    hi24, rho24 = O.split(x, 24)
    master = O.reconstruct(hi24, rho24, 24)
    fin = np.isfinite(master)
    mt = (master.view(np.uint32) & 0xFFFF) == 0x8000
    ref_m = torch.from_numpy(master.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    sel = fin & ~mt
    assert np.array_equal(hi24[sel], ref_m[sel])


def test_bf16_representable_values_have_zero_rho():
    bits = (np.arange(0, 1 << 16, dtype=np.uint32) << 16)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    for mb in (24, 32):
        hi, rho = O.split(x, mb)
        assert np.all(rho == 0)
        assert np.array_equal(hi.astype(np.uint32) << 16, x.view(np.uint32))


def test_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan,
                  np.finfo(np.float32).max, -np.finfo(np.float32).max,
                  np.finfo(np.float32).tiny, 1e-45], dtype=np.float32)
    for mb in (24, 32):
        hi, rho = O.split(x, mb)
        back = O.reconstruct(hi, rho, mb)
        assert np.array_equal(back[:4].view(np.uint32), x[:4].view(np.uint32))
        assert np.isnan(back[4]) and np.isnan(back[5]) and rho[4] == 0
    # FLT_MAX rounds past the largest 24-bit float: the master overflows to inf
    hi, rho = O.split(x[6:8], 24)
    assert np.all(np.isinf(O.reconstruct(hi, rho, 24)))
    hi, rho = O.split(x[6:8], 32)
    assert np.array_equal(O.reconstruct(hi, rho, 32), x[6:8])


def test_bad_master_bits():
    with pytest.raises(ValueError):
        O.split(np.zeros(4, np.float32), 16)


def test_exponent_sweep_statistics():
    """The harness' statistics for the reading (exact fraction, mean relative
    error); 32-bit master is exact everywhere, 24-bit within 2^-16."""
    x = W.exponent_sweep(random_sign=True).numpy()
    assert x.size == 64 * 65536
    hi, rho = O.split(x, 24)
    back = O.reconstruct(hi, rho, 24).astype(np.float64)
    rel = np.abs(back - x) / np.abs(x.astype(np.float64))
    assert 3e-6 < rel.mean() < 8e-6
    xs = W.exponent_sweep(random_sign=False).numpy()
    hi, rho = O.split(xs, 32)
    assert np.mean(O.reconstruct(hi, rho, 32) == xs) == 1.0
