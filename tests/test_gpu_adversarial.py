"""Adversarial value ranges through both decode scans, against the oracle.

The tensor-core scan regroups the dequantized arithmetic: codes enter the
tensor core as binary16 subnormals, q * scale and P * scale are split into
exact binary16 hi/lo pairs, q is scaled per head and P per pool by powers of
two chosen from the largest scales the pool has seen.  These are the places
where bits could be lost, so each case here drives one of them to its edge:
constant groups (scale 0), scales in the binary16 subnormal band, channels
whose scales span 1e-4 .. 1e2 inside one group, the x20 channel and x8 row
outliers together, q rows from 1e-3 to 1e3, and a pool whose largest INT2 K
and V scales grow after requests were already decoded.  Each case runs at
g = 4 and g = 8 over an INT2-only, an INT4-only and a mixed request, on both
scans; outputs must lie within max-abs 1e-3 and relative-L2 1e-4 of the fp64
oracle, and codes, scale/zero and tables must match it bit for bit.  The
same ranges run on INT3 and FP4 pages too."""
import numpy as np
import pytest

import oracle
from harness import assert_outputs_close, compare_content

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / np.sqrt(128)))
HKV = 2


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def bf16(x):
    """float array -> bf16 bits (round to nearest even)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def _dev(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).cuda()


class Pair:
    """A GPU pool and an oracle pool fed the same explicit bf16 rows."""

    def __init__(self, kvq, hkv, n_req, impl, n2=64, n4=64, max_tab=32, n3=0, nf=0):
        self.gpu = kvq.KVPool(hkv, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        self.gpu.set_decode_impl(impl)
        self.orc = oracle.OraclePool(hkv, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        self.g = [self.gpu.open() for _ in range(n_req)]
        self.o = [self.orc.open() for _ in range(n_req)]
        self.hkv = hkv

    def append(self, r, k, v, bits, chunk=96):
        kb, vb = bf16(k), bf16(v)
        for t0 in range(0, bits.size, chunk):
            sl = slice(t0, min(bits.size, t0 + chunk))
            n = sl.stop - sl.start
            self.gpu.append(_dev(kb[sl]), _dev(vb[sl]), np.full(n, self.g[r]), bits[sl])
            assert self.orc.append(np.full(n, self.o[r]), bits[sl], kb[sl], vb[sl]) == oracle.OK

    def reorder(self):
        self.gpu.reorder(self.g)
        assert self.orc.reorder(self.o) == oracle.OK
        self.gpu.sync()

    def check(self, q, what, reqs=None):
        reqs = list(range(len(self.g))) if reqs is None else reqs
        qb = bf16(q)
        out = self.gpu.decode(_dev(qb), [self.g[r] for r in reqs], SCALE)
        self.gpu.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all(), what
        ref = self.orc.decode(qb, [self.o[r] for r in reqs], SCALE).reshape(got.shape)
        for r in reqs:
            compare_content(self.gpu.export(self.g[r]), self.orc.export(self.o[r]), list(range(self.hkv)))
        return assert_outputs_close(got, ref, what)


def _base(rng, n, hkv=HKV):
    return rng.standard_normal((n, hkv, 128)).astype(np.float32)


def _three_requests(rng):
    """Bit widths of an INT2-only, an INT4-only and a mixed request."""
    return [np.full(256, 2, np.uint8), np.full(200, 4, np.uint8),
            np.where(rng.random(300) < 0.6, 2, 4).astype(np.uint8)]


def _constant_and_subnormal(rng, n):
    k, v = _base(rng, n), _base(rng, n)
    for x in (k, v):
        blocks = x.reshape(n, HKV, 4, 32)
        const = rng.random((n, HKV, 4)) < 0.3                 # per-token groups with scale 0
        blocks[const] = rng.standard_normal(int(const.sum()))[:, None]
        tiny = rng.random((n, HKV, 4)) < 0.15                 # groups whose scale is a binary16 subnormal
        blocks[tiny] *= 1e-5
    ch = rng.random((HKV, 128))
    k[:, ch < 0.15] = rng.standard_normal(int((ch < 0.15).sum()))   # channels constant over every page
    k[:, (ch >= 0.15) & (ch < 0.3)] *= 1e-5                         # channels with subnormal INT2 scales
    return k, v


def _mixed_channel_scales(rng, n):
    k, v = _base(rng, n), _base(rng, n)
    k *= 10.0 ** rng.uniform(-4, 2, (1, HKV, 128)).astype(np.float32)
    v *= 10.0 ** rng.uniform(-4, 2, (1, HKV, 128)).astype(np.float32)
    return k, v


def _extremes(rng, n):
    k, v = _base(rng, n), _base(rng, n)
    for h in range(HKV):
        k[:, h, rng.choice(128, 4, replace=False)] *= 20.0
    rows = rng.random(n) < 0.05
    k[rows] *= 8.0
    v[rows] *= 8.0
    return k, v


CASES = {"constant_and_subnormal": _constant_and_subnormal, "mixed_channel_scales": _mixed_channel_scales,
         "extremes": _extremes}


@pytest.mark.parametrize("impl", [1, 2])
@pytest.mark.parametrize("g", [4, 8])
@pytest.mark.parametrize("case", sorted(CASES))
def test_value_ranges(kvq, case, g, impl):
    rng = np.random.default_rng([7, g, len(case)])
    bits = _three_requests(rng)
    P = Pair(kvq, HKV, len(bits), impl)
    for r, b in enumerate(bits):
        k, v = CASES[case](rng, b.size)
        P.append(r, k, v, b)
    P.reorder()
    q = rng.standard_normal((len(bits), HKV * g, 128)).astype(np.float32)
    P.check(q, f"{case} g={g} impl={impl}")


@pytest.mark.parametrize("impl", [1, 2])
@pytest.mark.parametrize("g", [4, 8])
@pytest.mark.parametrize("case", sorted(CASES))
def test_value_ranges_int3_fp4(kvq, case, g, impl):
    """The same value ranges on INT3 and FP4 pages: an INT3-only, an FP4-only
    and a request mixing all four widths."""
    from mixed_precision_kv_gb300 import KV_WIDTH_FP4
    rng = np.random.default_rng([10, g, len(case)])
    bits = [np.full(200, 3, np.uint8), np.full(160, KV_WIDTH_FP4, np.uint8),
            rng.choice(np.array([2, 3, 4, KV_WIDTH_FP4], np.uint8), 300)]
    P = Pair(kvq, HKV, len(bits), impl, n3=32, nf=32)
    for r, b in enumerate(bits):
        k, v = CASES[case](rng, b.size)
        P.append(r, k, v, b)
    P.reorder()
    q = rng.standard_normal((len(bits), HKV * g, 128)).astype(np.float32)
    P.check(q, f"INT3/FP4 {case} g={g} impl={impl}")


@pytest.mark.parametrize("impl", [1, 2])
@pytest.mark.parametrize("g", [4, 8])
def test_query_magnitudes(kvq, g, impl):
    """q heads scaled by 1e3, 1, 1e-3 and 1e-2 in turn (the per-head power-of-two
    scaling of the q operands), over keys with x20 outlier channels."""
    rng = np.random.default_rng([8, g])
    bits = _three_requests(rng)
    P = Pair(kvq, HKV, len(bits), impl)
    for r, b in enumerate(bits):
        k, v = _extremes(rng, b.size)
        P.append(r, k, v, b)
    P.reorder()
    q = rng.standard_normal((len(bits), HKV * g, 128)).astype(np.float32)
    q *= np.array([1e3, 1.0, 1e-3, 1e-2] * (2 * g))[:HKV * g][None, :, None].astype(np.float32)
    P.check(q, f"q magnitudes g={g} impl={impl}")


@pytest.mark.parametrize("impl", [1, 2])
@pytest.mark.parametrize("g", [4, 8])
def test_pool_scale_maximum_grows_after_decode(kvq, g, impl):
    """Requests are decoded, then a new request's first INT2 page raises the
    largest INT2 K scale and the largest V scale the pool has seen (so the
    scans' power-of-two operand scales change); every request, old and new,
    must still match the oracle."""
    rng = np.random.default_rng([9, g])
    P = Pair(kvq, HKV, 3, impl)
    for r in range(2):
        b = np.where(rng.random(160) < 0.5, 2, 4).astype(np.uint8)
        k, v = _base(rng, b.size), _base(rng, b.size)
        P.append(r, k, v, b)
    P.reorder()
    q = rng.standard_normal((2, HKV * g, 128)).astype(np.float32)
    P.check(q, f"before growth g={g} impl={impl}", reqs=[0, 1])
    k, v = _base(rng, 64), _base(rng, 64)
    k[:32] *= 300.0                                           # its first INT2 page: K scales x300, V scales x20
    v[:32] *= 20.0                                            # (outputs stay O(10), inside fp32's 1e-3 reach)
    P.append(2, k, v, np.array([2] * 32 + [4] * 32, np.uint8))
    P.reorder()
    q = rng.standard_normal((3, HKV * g, 128)).astype(np.float32)
    P.check(q, f"after growth g={g} impl={impl}")
    P.check(q[:2], f"old requests after growth g={g} impl={impl}", reqs=[0, 1])
