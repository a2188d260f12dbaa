"""Pins of the oracle's group quantizer (TriAxialKV, key design 3)."""
import numpy as np
import pytest

from conftest import golden_lines


def _expand(field):
    body, _, rep = field.partition(" x")
    vals = [float(v) for v in body.split(",")]
    return vals * (int(rep) if rep else 1)


def _h2f(b):
    return np.array([b], np.uint16).view(np.float16).astype(np.float64)[0]


def _dequant_exact(codes, s_bits, z_bits):
    # code * s + z is exact in fp64 (all terms are multiples of 2^-24 below 2^17);
    # one rounding to fp32 then equals a correctly rounded fmaf.
    return (codes.astype(np.float64) * _h2f(s_bits) + _h2f(z_bits)).astype(np.float32)


def test_golden_cases(orc):
    n = 0
    for ln in golden_lines("quant_cases.txt"):
        name, bits, vals, meta, codes = [f.strip() for f in ln.split("|")]
        x = np.array(_expand(vals), np.float32)
        want = np.array(_expand(codes), np.uint8)
        s_hex, z_hex = meta.split()
        c, s, z = orc.quant_group(x, int(bits))
        assert (s, z) == (int(s_hex, 16), int(z_hex, 16)), name
        assert np.array_equal(c, want), name
        n += 1
    assert n == 6


def _groups(rng, n_groups, n=32):
    kinds = []
    for i in range(n_groups):
        k = i % 6
        x = rng.standard_normal(n).astype(np.float32)
        if k == 1:
            x *= 20.0
        elif k == 2:
            x = (x * 1e-3 + 7.0).astype(np.float32)          # tiny range, large offset
        elif k == 3:
            x = (x * 3e-6).astype(np.float32)                 # scale in the binary16 subnormal band
        elif k == 4:
            x = (x * 3000.0).astype(np.float32)
        elif k == 5:
            x[rng.integers(0, n)] *= 500.0                    # one outlier
        kinds.append(x.astype(np.float32))
    return kinds


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_are_nearest_levels(orc, bits):
    """Brute force over all 2^b codes: the chosen level is the nearest one,
    up to the two fp32 roundings in (x - z) / s."""
    rng = np.random.default_rng(10 + bits)
    qmax = (1 << bits) - 1
    for x in _groups(rng, 600):
        c, s, z = orc.quant_group(x, bits)
        if s == 0:
            assert (c == 0).all()
            continue
        levels = _dequant_exact(np.arange(qmax + 1), s, z).astype(np.float64)
        err = np.abs(x.astype(np.float64)[:, None] - levels[None, :])
        chosen = err[np.arange(x.size), c]
        sf = _h2f(s)
        u = np.abs((x.astype(np.float64) - _h2f(z)) / sf)
        slack = 4 * 2.0 ** -23 * np.maximum(u, 1.0) * sf + 2.0 ** -149
        assert (chosen <= err.min(axis=1) + slack).all()
        # dequantization = fmaf(code, s, z)
        xh = np.array([orc.dequant(ci, s, z) for ci in c], np.float32)
        assert np.array_equal(xh, _dequant_exact(c, s, z))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_roundtrip_error_bound(orc, bits):
    """|x - x^| <= s/2 inside the covered range; outside it the excess is bounded
    by the binary16 rounding of the zero and of the scale."""
    rng = np.random.default_rng(20 + bits)
    qmax = (1 << bits) - 1
    for x in _groups(rng, 600):
        c, s, z = orc.quant_group(x, bits)
        xd = x.astype(np.float64)
        xh = _dequant_exact(c, s, z).astype(np.float64)
        sf, zf = _h2f(s), _h2f(z)
        ulp = np.spacing(np.abs(xh).astype(np.float32)).astype(np.float64)
        inside = (xd >= zf - sf / 2) & (xd <= zf + (qmax + 0.5) * sf)
        assert (np.abs(xd - xh)[inside] <= sf / 2 * (1 + 2.0 ** -20) + 2 * ulp[inside]).all()
        s_exact = (xd.max() - xd.min()) / qmax
        excess = abs(xd.min() - zf) + qmax * abs(s_exact - sf)
        assert (np.abs(xd - xh) <= sf / 2 + excess + 2 * ulp + 1e-30).all()


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_exact_grid_roundtrip(orc, bits):
    """Values on a grid z + c*s with binary16-exact s, z and codes 0 and 2^b-1
    present: the quantizer must return exactly that s, z and those codes."""
    rng = np.random.default_rng(30 + bits)
    qmax = (1 << bits) - 1
    for _ in range(300):
        s = int(rng.integers(1, 1024)) * 2.0 ** -6
        z = int(rng.integers(-512, 513)) * 2.0 ** -6
        codes = rng.integers(0, qmax + 1, 32)
        codes[rng.integers(0, 32)] = 0
        codes[rng.integers(0, 32)] = qmax
        if codes.min() != 0 or codes.max() != qmax:
            continue
        x = (codes * s + z).astype(np.float32)
        c, sb, zb = orc.quant_group(x, bits)
        assert _h2f(sb) == s and _h2f(zb) == z
        assert np.array_equal(c, codes.astype(np.uint8))


def test_constant_group_and_range_errors(orc):
    for v in (0.0, -3.25, 1e-6, 65504.0):
        c, s, z = orc.quant_group(np.full(32, v, np.float32), 4)
        assert s == 0 and (c == 0).all()
        assert z == int(np.float16(v).view(np.uint16))
    with pytest.raises(orc.OracleError) as e:
        orc.quant_group(np.array([0.0] * 31 + [65520.0], np.float32), 4)
    assert e.value.code == orc.RANGE
    with pytest.raises(orc.OracleError):
        orc.quant_group(np.array([np.nan] + [0.0] * 31, np.float32), 2)
