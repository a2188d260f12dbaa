"""Pins of the oracle's binary16 converter (scale/zero storage format)."""
import numpy as np

from conftest import golden_lines


def test_golden_edge_table(orc):
    rows = [ln.split()[:2] for ln in golden_lines("f16_edges.txt")]
    x = np.array([int(a, 16) for a, _ in rows], dtype=np.uint32).view(np.float32)
    want = np.array([int(b, 16) for _, b in rows], dtype=np.uint16)
    assert np.array_equal(orc.f32_to_f16(x), want)


def test_exhaustive_low_bits_against_numpy_in_the_rounding_band(orc):
    # Float32 exponent fields [100, 143] (2^-27 .. 2^17), both signs: every
    # pattern of the low 16 fraction bits (which decide the rounding, ties and
    # the carry) under 32 random patterns of the high 7 bits, plus the all-zero
    # and all-one high bits.  Covers subnormals, ties and the overflow edge.
    rng = np.random.default_rng(3)
    low = np.arange(1 << 16, dtype=np.uint32)
    for sign in (0, 1):
        for ef in range(100, 144):
            highs = np.concatenate([[0, 0x7F], rng.integers(0, 128, 32)]).astype(np.uint32)
            bits = ((highs[:, None] << np.uint32(16)) | low[None, :]).ravel()
            bits = bits | np.uint32(ef << 23) | np.uint32(sign << 31)
            x = bits.view(np.float32)
            got = orc.f32_to_f16(x)
            want = x.astype(np.float16).view(np.uint16)
            assert np.array_equal(got, want), (sign, ef)


def test_far_ranges_and_roundtrip(orc):
    rng = np.random.default_rng(1)
    small = (rng.integers(0, 100 << 23, 1 << 20, dtype=np.uint64).astype(np.uint32))
    big = (rng.integers(144 << 23, 255 << 23, 1 << 20, dtype=np.uint64).astype(np.uint32))
    for b in (small, big, small | np.uint32(1 << 31), big | np.uint32(1 << 31)):
        x = b.view(np.float32)
        assert np.array_equal(orc.f32_to_f16(x), x.astype(np.float16).view(np.uint16))
    h = np.arange(1 << 16, dtype=np.uint16)
    finite = (h & 0x7C00) != 0x7C00
    back = orc.f16_to_f32(h)
    assert np.array_equal(back[finite], h[finite].view(np.float16).astype(np.float32))
    assert np.array_equal(orc.f32_to_f16(back[finite]), h[finite])
