"""Oracle pins for FP4 (E2M1) pages (TriAxialKV, limitations and outlook:
non-uniform FP formats; the pages' uniform FP4 baseline; HyQuant background:
s = max|X| / c_B).  What fixes the results: the E2M1 value table of the
format's definition, hand-worked groups (tests/golden/fp4_cases.txt),
brute force over all 16 codes, closed forms of ids and table order, the
numpy restatement of attention from the export, and an all-FP4 request
against an independently written per-token FP4 attention."""
import numpy as np
import pytest

import kvsynth
from conftest import golden_lines
from np_ref import attention_from_export, quant_fp4_tokens_np

SCALE = float(np.float32(1 / np.sqrt(128)))
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # the format's magnitudes by code bits 0..2


def _expand(field):
    out = []
    for part in field.split():
        if part.startswith("x"):
            out = out * int(part[1:])
        else:
            out += [float(v) for v in part.split(",")]
    return out


def test_e2m1_table(orc):
    for c in range(16):
        assert orc.e2m1_value(c) == (-1.0 if c & 8 else 1.0) * E2M1[c & 7]


def test_golden_cases(orc):
    n = 0
    for ln in golden_lines("fp4_cases.txt"):
        name, vals, s_hex, codes = [f.strip() for f in ln.split("|")]
        x = np.array(_expand(vals), np.float32)
        c, s = orc.fp4_group(x)
        assert s == int(s_hex, 16), name
        assert np.array_equal(c, np.array(_expand(codes), np.uint8)), name
        n += 1
    assert n == 6


def _groups(rng, n_groups, n=32):
    out = []
    for i in range(n_groups):
        x = rng.standard_normal(n).astype(np.float32)
        k = i % 5
        if k == 1:
            x *= 20.0
        elif k == 2:
            x = (x * 3e-6).astype(np.float32)            # scale in the binary16 subnormal band
        elif k == 3:
            x[rng.integers(0, n)] *= 500.0                # one outlier
        elif k == 4:
            x = (x * 3000.0).astype(np.float32)
        out.append(x.astype(np.float32))
    return out


def test_codes_are_nearest_values_with_even_ties(orc):
    """Brute force over the 16 codes: the chosen value is the nearest to
    x / s (fp32 quotient), ties to the even mantissa, and the scale is the
    binary16 rounding of max|x| / 6."""
    rng = np.random.default_rng(44)
    grid = np.array([(-1.0 if c & 8 else 1.0) * E2M1[c & 7] for c in range(16)])
    for x in _groups(rng, 300):
        c, s = orc.fp4_group(x)
        sf = np.float32(np.uint16(s).view(np.float16))
        assert s == np.float16(np.float32(np.abs(x).max()) / np.float32(6.0)).view(np.uint16)
        if sf == 0:
            assert not c.any()
            continue
        u = (x / sf).astype(np.float32).astype(np.float64)
        for ui, ci in zip(u, c):
            d = np.abs(grid - ui)
            best = np.flatnonzero(d == d.min())
            if ci & 7 == 0:
                assert ci == 0                            # zero is +0
                assert np.any((np.array(best) & 7) == 0)
            else:
                assert ci in best
                if best.size > 1:
                    assert (ci & 1) == 0                  # a tie takes the even mantissa


def test_reconstruction_bound_and_saturation(orc):
    """|x - s v| is at most half the grid step around x / s (times s), and
    values beyond 6 s (s rounded down) saturate to 6 s."""
    rng = np.random.default_rng(45)
    for x in _groups(rng, 200):
        c, s = orc.fp4_group(x)
        sf = float(np.uint16(s).view(np.float16))
        if sf == 0:
            continue
        v = np.array([orc.e2m1_value(ci) for ci in c])
        a = np.abs(x.astype(np.float64)) / sf
        step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
        over = a > 6.0
        assert np.all(np.abs(np.abs(v[~over]) - a[~over]) <= step[~over] / 2 + 1e-6)
        assert np.all(np.abs(v[over]) == 6.0)


def _kv(n, hkv, stream, seed=5, tok0=0):
    return (kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_K, stream, tok0),
            kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_V, stream, tok0))


def test_routing_ids_and_reorder(orc):
    """n2 = 4, n4 = 8, n3 = 4, nf = 8: INT4 ids [4, 12), INT3 [12, 16), FP4 [16, 24)."""
    P = orc.OraclePool(1, 4, 8, 1, 16, n_int3_pages=4, n_fp4_pages=8)
    r = P.open()
    bits = np.array([orc.FP4] * 40 + [4] * 3 + [3] * 2 + [2] * 32, np.uint8)
    k, v = _kv(bits.size, 1, 0)
    assert P.append(np.full(bits.size, r), bits, k, v) == orc.OK
    ex = P.export(r, content=False)
    assert ex["ids"].tolist() == [16, 17, 4, 12, 0]      # FP4 16 (32), 17 (8); INT4 4; INT3 12; staging 5 -> INT2 0
    assert ex["fill"].tolist() == [32, 8, 3, 2, 32]
    assert P.reorder([r]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [0, 12, 4, 16, 17]


def test_decode_brute_force_with_fp4_pages(orc):
    rng = np.random.default_rng(3)
    P = orc.OraclePool(2, 32, 32, 2, 64, n_int3_pages=32, n_fp4_pages=32)
    rids, q = [], kvsynth.fill_bf16_host(2, 8, 128, 9, kvsynth.TENSOR_Q, 0)
    for i, m in enumerate([150, 77]):
        r = P.open()
        k, v = _kv(m, 2, i)
        bits = rng.choice(np.array([2, 3, 4, orc.FP4], np.uint8), m)
        assert P.append(np.full(m, r), bits, k, v) == orc.OK
        ev = rng.choice(m, m // 5, replace=False)
        assert P.evict(np.full(ev.size, r), ev) == orc.OK
        rids.append(r)
    out = P.decode(q, rids, SCALE)
    for b, r in enumerate(rids):
        ex = P.export(r)
        fp4 = ex["ids"] >= 32 + 32 + 32                    # FP4 ids follow the INT2, INT4 and INT3 ids
        assert fp4.any()
        for hq in range(8):
            ref = attention_from_export(ex, hq // 4, kvsynth.bf16_to_f32(q[b, hq]), SCALE, fp4_pages=fp4)
            np.testing.assert_allclose(out[b * 8 + hq], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(P.decode(q, rids, SCALE, n_splits=7), out, rtol=1e-12, atol=1e-14)


def test_all_fp4_equals_uniform_per_token_fp4_attention(orc):
    n = 210
    P = orc.OraclePool(2, 4, 4, 1, 16, n_fp4_pages=16)
    r = P.open()
    k, v = _kv(n, 2, 4)
    assert P.append(np.full(n, r), np.full(n, orc.FP4, np.uint8), k, v) == orc.OK
    q = kvsynth.fill_bf16_host(1, 8, 128, 9, kvsynth.TENSOR_Q, 0)
    out = P.decode(q, [r], SCALE)
    for hq in range(8):
        kv = hq // 4
        K = quant_fp4_tokens_np(kvsynth.bf16_to_f32(k[:, kv])).astype(np.float64)
        V = quant_fp4_tokens_np(kvsynth.bf16_to_f32(v[:, kv])).astype(np.float64)
        lg = SCALE * (K @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out[hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-13)


def test_fp4_oom_and_invalid(orc):
    P = orc.OraclePool(1, 2, 2, 1, 8, n_fp4_pages=1)
    r = P.open()
    k, v = _kv(33, 1, 7)
    assert P.append(np.full(33, r), np.full(33, orc.FP4, np.uint8), k, v) == orc.OOM
    assert P.info(r) == (0, 0)
    assert P.append(np.full(1, r), np.array([0xF3], np.uint8), k[:1], v[:1]) == orc.INVALID
    Q = orc.OraclePool(1, 2, 2, 1, 8)
    s = Q.open()
    assert Q.append(np.full(1, s), np.array([orc.FP4], np.uint8), k[:1], v[:1]) == orc.OOM   # no FP4 pages
