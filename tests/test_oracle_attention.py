"""Pins of the oracle's decode attention (TriAxialKV key design 4; HyQuant
online softmax and Algorithm 3 split-K merge; IntentKV sentinel dead slot)."""
import numpy as np
import pytest

import kvsynth
from np_ref import attention_from_export, quant_int4_tokens_np

SCALE = float(np.float32(1 / np.sqrt(128)))


def _build(orc, ns, bits_fn, hkv=2, seed=5, evict_frac=0.0, rng=None, sel=None):
    """One request per entry of ns; returns (pool, req ids, per-request k/v bf16)."""
    rng = rng or np.random.default_rng(seed)
    P = orc.OraclePool(hkv, 256, 256, len(ns), 256, sel_heads=sel)
    sel = P.sel
    rids, kvs = [], []
    for i, n in enumerate(ns):
        r = P.open()
        k = kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_K, i)
        v = kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_V, i)
        bits = bits_fn(n, rng)
        assert P.append(np.full(n, r), bits, k[:, sel], v[:, sel]) == orc.OK
        if evict_frac and n:
            ev = rng.choice(n, int(evict_frac * n), replace=False)
            assert P.evict(np.full(ev.size, r), ev) == orc.OK
        rids.append(r)
        kvs.append((k, v, bits))
    return P, rids, kvs


def _mixed(n, rng):
    return np.where(rng.random(n) < 0.55, 2, 4).astype(np.uint8)


def _q(B, Hq, seed=9):
    return kvsynth.fill_bf16_host(B, Hq, 128, seed, kvsynth.TENSOR_Q, 0)


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 64])
def test_brute_force_small(orc, n):
    P, rids, _ = _build(orc, [n, 64 - n + 1], _mixed, evict_frac=0.2)
    q = _q(2, 8)
    out = P.decode(q, rids, SCALE)
    for b, r in enumerate(rids):
        ex = P.export(r)
        for hq in range(8):
            ref = attention_from_export(ex, hq // 4, kvsynth.bf16_to_f32(q[b, hq]), SCALE)
            np.testing.assert_allclose(out[b * 8 + hq], ref, rtol=1e-12, atol=1e-13)


def test_page_order_and_split_invariance(orc):
    rng = np.random.default_rng(11)
    P, rids, _ = _build(orc, [700, 300], _mixed, evict_frac=0.05, rng=rng)
    q = _q(2, 8)
    base = P.decode(q, rids, SCALE)
    for s in (2, 3, 7, 64, 5000):
        np.testing.assert_allclose(P.decode(q, rids, SCALE, n_splits=s), base, rtol=1e-12, atol=1e-14)
    assert P.reorder(rids) == orc.OK
    np.testing.assert_allclose(P.decode(q, rids, SCALE), base, rtol=1e-12, atol=1e-14)


def test_all_int4_equals_uniform_per_token_int4_attention(orc):
    """Budget B = 4: every token is INT4, and the output equals plain softmax
    attention over an independently written per-token INT4 quantization."""
    n = 333
    P, rids, kvs = _build(orc, [n], lambda n, r: np.full(n, 4, np.uint8))
    q = _q(1, 8)
    out = P.decode(q, rids, SCALE)
    k, v, _ = kvs[0]
    for hq in range(8):
        kv = hq // 4
        K = quant_int4_tokens_np(kvsynth.bf16_to_f32(k[:, kv])).astype(np.float64)
        V = quant_int4_tokens_np(kvsynth.bf16_to_f32(v[:, kv])).astype(np.float64)
        lg = SCALE * (K @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out[hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-13)


def test_eviction_equals_deletion_and_all_dead_is_zero(orc):
    n = 200
    rng = np.random.default_rng(13)
    ev = np.sort(rng.choice(n, 37, replace=False))
    keep = np.setdiff1d(np.arange(n), ev)
    k = kvsynth.fill_bf16_host(n, 2, 128, 3, kvsynth.TENSOR_K, 0)
    v = kvsynth.fill_bf16_host(n, 2, 128, 3, kvsynth.TENSOR_V, 0)
    q = _q(1, 8)
    P = orc.OraclePool(2, 64, 64, 2, 64)
    r = P.open()
    assert P.append(np.full(n, r), np.full(n, 4, np.uint8), k, v) == orc.OK
    assert P.evict(np.full(ev.size, r), ev) == orc.OK
    Q = orc.OraclePool(2, 64, 64, 1, 64)
    s = Q.open()
    assert Q.append(np.full(keep.size, s), np.full(keep.size, 4, np.uint8), k[keep], v[keep]) == orc.OK
    np.testing.assert_allclose(P.decode(q, [r], SCALE), Q.decode(q, [s], SCALE), rtol=1e-12, atol=1e-14)
    assert P.evict(np.full(n, r), np.arange(n)) == orc.OK
    assert np.array_equal(P.decode(q, [r], SCALE), np.zeros((8, 128)))
    e = P.open()
    assert np.array_equal(P.decode(q, [e], SCALE), np.zeros((8, 128)))


def test_textbook_limit_fine_grid(orc):
    """K and V on an exact INT4 grid (every 32-channel group spans 0..15 times a
    binary16 scale): quantization is lossless, so the oracle must equal plain
    softmax attention of the bf16 inputs."""
    rng = np.random.default_rng(17)
    n, hkv = 96, 1
    codes_k = rng.integers(0, 16, (n, 128))
    codes_v = rng.integers(0, 16, (n, 128))
    for c in (codes_k, codes_v):
        c[:, 0::32] = 0
        c[:, 1::32] = 15
    Kx = (codes_k * 0.125 - 1.0).astype(np.float32)
    Vx = (codes_v * 0.25 + 0.5).astype(np.float32)
    to_bf = lambda x: (x.view(np.uint32) >> 16).astype(np.uint16).reshape(n, hkv, 128)
    P = orc.OraclePool(hkv, 8, 8, 1, 8)
    r = P.open()
    assert P.append(np.full(n, r), np.full(n, 4, np.uint8), to_bf(Kx), to_bf(Vx)) == orc.OK
    q = _q(1, 4)
    out = P.decode(q, [r], SCALE)
    for hq in range(4):
        lg = SCALE * (Kx.astype(np.float64) @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out[hq], (w @ Vx.astype(np.float64)) / w.sum(), rtol=1e-12, atol=1e-13)
