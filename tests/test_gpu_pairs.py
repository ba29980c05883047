"""GPU parity of the two standalone kernel pairs against the CPU oracle, through
the C ABI: codes, fp16 scales, dequantized values, theta', rho and the
reconstructed master must be identical bit for bit."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_state_optimizer_gb300 as fo
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
SPECS = ["momentum", "variance", "momentum_linear", "variance_linear"]


def gpu_quantize(x: np.ndarray, spec: str):
    n = x.size
    signed = spec.startswith("momentum")
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    codes = torch.empty(n, dtype=torch.int8 if signed else torch.uint8, device=DEV)
    scales = torch.empty(max(fo.n_groups(n), 1), dtype=torch.float16, device=DEV)
    fo.fo_quantize(xd, spec, codes, scales)
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    fo.fo_dequantize(codes, scales, spec, out)
    torch.cuda.synchronize()
    return (codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)[: fo.n_groups(n)],
            out.cpu().numpy())


def same_f32(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


@pytest.mark.parametrize("spec", SPECS)
def test_quantize_battery_bit_exact(spec):
    for name, t in W.battery().items():
        x = t.numpy()
        if spec.startswith("variance"):
            x = np.abs(x)
        c, s, d = gpu_quantize(x, spec)
        rc, rs = O.quantize(x, spec)
        assert np.array_equal(c, rc), (name, spec, np.mean(c == rc))
        assert np.array_equal(s, rs), (name, spec)
        assert same_f32(d, O.dequantize(rc, rs, spec)), (name, spec)
        # the harness' agreement metrics, for the record
        agree = float(np.mean(c == rc))
        within1 = float(np.mean(np.abs(c.astype(int) - rc.astype(int)) <= 1))
        assert agree == 1.0 and within1 == 1.0


@pytest.mark.parametrize("n", [1, 15, 16, 17, 31, 32, 33, 63, 4095, 4096, 4097, 65553, (1 << 20) + 5])
def test_quantize_ragged_sizes(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * np.exp(2 * rng.standard_normal(n))).astype(np.float32)
    for spec in SPECS:
        xin = np.abs(x) if spec.startswith("variance") else x
        c, s, d = gpu_quantize(xin, spec)
        rc, rs = O.quantize(xin, spec)
        assert np.array_equal(c, rc) and np.array_equal(s, rs), (n, spec)
        assert same_f32(d, O.dequantize(rc, rs, spec))


def _boundary_inputs(spec: str) -> np.ndarray:
    """Groups whose first element fixes the scale at exactly 1.0 and whose other
    elements sit on, and a few ulps around, the inputs where the code argument
    is exactly k + 1/2 (round-half-even territory): every one of them must
    take the exact path and still agree with the oracle."""
    out = []
    ks = np.arange(0, 127) if spec.startswith("momentum") else np.arange(0, 255)
    for k in ks:
        if spec == "momentum":
            z = (k + 0.5) / 127.0
            x0 = z / (2.0 - z)            # inverse softsign at scale 1
        elif spec == "variance":
            x0 = ((k + 0.5) / 255.0) ** 2  # inverse of 255 sqrt(v)
        elif spec == "momentum_linear":
            x0 = (k + 0.5) / 127.0
        else:
            x0 = (k + 0.5) / 255.0
        x0 = np.float32(x0)
        nb = [np.float32(np.nextafter(x0, np.float32(np.inf * d))) for d in (1, -1)]
        cand = [x0, nb[0], nb[1], np.float32(np.nextafter(nb[0], np.float32(np.inf))),
                np.float32(np.nextafter(nb[1], np.float32(-np.inf)))]
        g = np.zeros(32, np.float32)
        g[0] = 1.0
        g[1:1 + len(cand)] = cand
        if spec.startswith("momentum"):
            g[8:8 + len(cand)] = [-c for c in cand]
        out.append(g)
    return np.concatenate(out)


@pytest.mark.parametrize("spec", SPECS)
def test_quantize_half_code_boundaries(spec):
    x = _boundary_inputs(spec)
    c, s, d = gpu_quantize(x, spec)
    rc, rs = O.quantize(x, spec)
    assert np.array_equal(s, rs)
    assert np.array_equal(c, rc), np.flatnonzero(c != rc)[:10]


@pytest.mark.parametrize("spec", SPECS)
def test_quantize_volume_heavy_tailed(spec):
    """4M values over many orders of magnitude, with zeros, subnormals and
    groups whose maximum is tiny or huge: the certified codes and their exact
    fallback against the oracle, and the dequantized values."""
    rng = np.random.default_rng(11)
    n = (1 << 22) + 9
    x = (rng.standard_normal(n) * np.exp(4 * rng.standard_normal(n))).astype(np.float32)
    x[::97] = 0.0
    x[5::101] = np.float32(3e-39)
    x[7::4099] *= np.float32(1e30)
    x[11::8191] = np.float32(2e-30)
    x = np.clip(x, -3e38, 3e38).astype(np.float32)
    if spec.startswith("variance"):
        x = np.abs(x)
    x = np.concatenate([x, _boundary_inputs(spec)])
    c, s, d = gpu_quantize(x, spec)
    rc, rs = O.quantize(x, spec)
    assert np.array_equal(s, rs), spec
    assert np.array_equal(c, rc), (spec, np.flatnonzero(c != rc)[:10])
    assert same_f32(d, O.dequantize(rc, rs, spec)), spec


def test_quantize_does_not_write_past_n():
    n = 4097
    x = torch.randn(n, device=DEV)
    codes = torch.full((n + 64,), 99, dtype=torch.int8, device=DEV)
    scales = torch.full((fo.n_groups(n) + 8,), 7.0, dtype=torch.float16, device=DEV)
    fo.fo_quantize(x, "momentum", codes, scales)
    torch.cuda.synchronize()
    assert torch.all(codes[n:] == 99)
    assert torch.all(scales[fo.n_groups(n):] == 7.0)


def test_empty_is_noop():
    x = torch.empty(0, device=DEV)
    fo.fo_quantize(x, "momentum", torch.empty(0, dtype=torch.int8, device=DEV),
                   torch.empty(0, dtype=torch.float16, device=DEV))


def test_misaligned_pointer_is_rejected():
    x = torch.zeros(64, device=DEV)
    codes = torch.zeros(80, dtype=torch.int8, device=DEV)
    scales = torch.zeros(8, dtype=torch.float16, device=DEV)
    with pytest.raises(fo.FoError, match="MISALIGNED"):
        fo.fo_quantize(x, "momentum", codes[1:65], scales)


def gpu_split(x: np.ndarray, rho_bits: int):
    n = x.size
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    hi = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    rho = torch.empty(n, dtype=torch.int8 if rho_bits == 8 else torch.int16, device=DEV)
    fo.fo_split(xd, rho_bits, hi, rho)
    back = torch.empty(n, dtype=torch.float32, device=DEV)
    fo.fo_reconstruct(hi, rho, rho_bits, back)
    torch.cuda.synchronize()
    return hi.cpu().view(torch.int16).numpy().view(np.uint16), rho.cpu().numpy(), back.cpu().numpy()


@pytest.mark.parametrize("rho_bits", [8, 16])
@pytest.mark.parametrize("sign", [True, False])
def test_split_exponent_sweep_bit_exact(rho_bits, sign):
    x = W.exponent_sweep(random_sign=sign).numpy()
    hi, rho, back = gpu_split(x, rho_bits)
    mb = 24 if rho_bits == 8 else 32
    rhi, rrho = O.split(x, mb)
    assert np.array_equal(hi, rhi) and np.array_equal(rho, rrho)
    assert np.array_equal(back.view(np.uint32), O.reconstruct(rhi, rrho, mb).view(np.uint32))
    if rho_bits == 16:
        assert np.array_equal(back.view(np.uint32), x.view(np.uint32))  # exact fraction 1.0
    else:
        rel = np.abs(back.astype(np.float64) - x) / np.abs(x.astype(np.float64))
        assert rel.max() <= 2.0 ** -16


@pytest.mark.parametrize("n", [1, 7, 16, 17, 4097])
def test_split_ragged_and_special(n):
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, np.finfo(np.float32).max,
                         -np.finfo(np.float32).max, 1e-45, -1e-40], dtype=np.float32)
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n).astype(np.float32)
    x[: min(n, specials.size)] = specials[: min(n, specials.size)]
    for rho_bits, mb in ((8, 24), (16, 32)):
        hi, rho, back = gpu_split(x, rho_bits)
        rhi, rrho = O.split(x, mb)
        assert np.array_equal(hi, rhi) and np.array_equal(rho, rrho)
        assert same_f32(back, O.reconstruct(rhi, rrho, mb))


def test_split16_round_trip_all_2_32_patterns():
    """Property at full range: every fp32 pattern reconstructs exactly with the
    32-bit master (NaN to NaN); the 24-bit master stays within 2^-16."""
    chunk = 1 << 28
    hi = torch.empty(chunk, dtype=torch.bfloat16, device=DEV)
    r16 = torch.empty(chunk, dtype=torch.int16, device=DEV)
    r8 = torch.empty(chunk, dtype=torch.int8, device=DEV)
    back = torch.empty(chunk, dtype=torch.float32, device=DEV)
    for start in range(0, 1 << 32, chunk):
        b64 = torch.arange(start, start + chunk, dtype=torch.int64, device=DEV)
        bits = torch.where(b64 >= 2 ** 31, b64 - 2 ** 32, b64).to(torch.int32)  # in range: no wrap
        x = bits.view(torch.float32)
        fo.fo_split(x, 16, hi, r16)
        fo.fo_reconstruct(hi, r16, 16, back)
        nan = torch.isnan(x)
        assert torch.equal(back.view(torch.int32)[~nan], bits[~nan]), hex(start)
        assert bool(torch.isnan(back[nan]).all())
        fo.fo_split(x, 8, hi, r8)
        fo.fo_reconstruct(hi, r8, 8, back)
        # normal range only: in the subnormal range the 24-bit master keeps a fixed
        # absolute spacing of 2^-141, so the relative bound does not apply there
        fin = torch.isfinite(x) & torch.isfinite(back) & (x.abs() >= 2.0 ** -126)
        rel = ((back[fin].double() - x[fin].double()).abs() / x[fin].double().abs())
        assert float(rel.max()) <= 2.0 ** -16, hex(start)
