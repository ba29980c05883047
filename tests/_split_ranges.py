"""Range workers of the exhaustive split pins (tests/test_oracle_split.py),
in a module of their own so that spawned pool workers import only numpy and
the oracle."""

import numpy as np

import oracle as O


def round_to_master24_f64(x: np.ndarray) -> np.ndarray:
    """Nearest 24-bit float (15 fraction bits), ties away from zero, in binary64
    arithmetic: multiples of 2^(E-15) for |x| in [2^E, 2^(E+1)), E >= -126;
    the fp32 subnormal range keeps the spacing 2^-141."""
    a = np.abs(np.asarray(x, dtype=np.float32).astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # guard floor(log2()) at binade edges
    e = np.where(2.0 ** e > a, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= a, e + 1, e)
    e = np.maximum(e, -126)
    ulp = 2.0 ** (e - 15)
    q = np.floor(a / ulp + 0.5) * ulp
    q = np.where(q >= 2.0 ** 128, np.inf, q)
    return np.copysign(q, np.asarray(x, dtype=np.float64))


def _round_trip32_range(lo: int, hi: int) -> str | None:
    """Check the 32-bit master round trip over bit patterns [lo, hi); returns a
    failure message or None (run in a worker process)."""
    chunk = 1 << 24
    for start in range(lo, hi, chunk):
        bits = np.arange(start, min(start + chunk, hi), dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        hi_, rho = O.split(x, 32)
        back = O.reconstruct(hi_, rho, 32).view(np.uint32)
        bad = np.flatnonzero(back != bits)  # only NaN patterns may come back changed
        if not (np.all(np.isnan(x[bad])) and np.all(np.isnan(back[bad].view(np.float32)))):
            return f"{hex(start)}: {bad[:5]}"
    return None


def _master24_stride_range(lo: int, hi: int) -> str | None:
    bits = np.arange(lo, hi, 97, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    hi_, rho = O.split(x, 24)
    back = O.reconstruct(hi_, rho, 24).astype(np.float64)
    if not np.array_equal(back, round_to_master24_f64(x)):
        return hex(lo)
    return None
