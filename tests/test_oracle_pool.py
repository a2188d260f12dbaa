"""Pins of the oracle's pool model: routing, page ids, reorder, eviction, repack
(TriAxialKV key designs 3-4; IntentKV layout-preserving eviction)."""
import numpy as np
import pytest

import kvsynth
from np_ref import dequant_page


def _kv(n, hkv, stream, seed=77):
    k = kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_K, stream)
    v = kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_V, stream)
    return k, v


def test_routing_closed_forms(orc):
    rng = np.random.default_rng(1)
    for trial in range(30):
        n = int(rng.integers(1, 400))
        bits = np.where(rng.random(n) < rng.random(), 2, 4).astype(np.uint8)
        P = orc.OraclePool(2, 64, 64, 2, 64)
        r = P.open()
        assert P.append(np.full(n, r), bits) == orc.OK
        ex = P.export(r, content=False)
        n2, n4 = int((bits == 2).sum()), int((bits == 4).sum())
        int2 = ex["is_int2"] == 1
        assert int(int2.sum()) == n2 // 32
        assert (ex["fill"][int2] == 32).all()
        assert (ex["ids"][int2] < 64).all() and (ex["ids"][~int2] >= 64).all()
        # INT4 pages: ceil(n4/32) tail pages plus one staging page when n2 % 32 > 0
        assert int((~int2).sum()) == -(-n4 // 32) + (1 if n2 % 32 else 0)
        assert int(ex["fill"].astype(int).sum()) == n
        assert (ex["live"] == (np.left_shift(1, ex["fill"].astype(np.int64)) - 1).astype(np.uint32)).all()


def test_lowest_free_ids_and_deferred_free(orc):
    P = orc.OraclePool(1, 8, 8, 4, 16)
    a = P.open()
    # 64 INT2-tagged tokens in one call: staging 8 fills, repacks to INT2 id 0;
    # the second staging page must be 9 (8 is only reusable after the call).
    assert P.append(np.full(64, a), np.full(64, 2, np.uint8)) == orc.OK
    assert P.export(a, content=False)["ids"].tolist() == [0, 1]
    b = P.open()
    assert P.append(np.full(1, b), np.full(1, 4, np.uint8)) == orc.OK
    assert P.export(b, content=False)["ids"].tolist() == [8]
    P.close_request(a)
    c = P.open()
    assert c == a
    assert P.append(np.full(33, c), np.array([2] * 32 + [4], np.uint8)) == orc.OK
    # staging takes 9 (lowest free INT4 id); at 32 tokens it is replaced in the
    # table by INT2 id 0; the b4 token then opens a tail page at 10 (9 only
    # becomes free again when the call ends).
    assert P.export(c, content=False)["ids"].tolist() == [0, 10]


def test_reorder_is_stable_int2_first(orc):
    rng = np.random.default_rng(2)
    P = orc.OraclePool(1, 200, 200, 3, 400)
    rs = [P.open() for _ in range(3)]
    for _ in range(6):
        req = rng.choice(rs, 300)
        bits = np.where(rng.random(300) < 0.6, 2, 4).astype(np.uint8)
        assert P.append(req, bits) == orc.OK
    for r in rs:
        before = P.export(r, content=False)["ids"].tolist()
        assert P.reorder([r]) == orc.OK
        after = P.export(r, content=False)["ids"].tolist()
        assert after == sorted(before, key=lambda i: i >= 200)       # Python's sort is stable
        k = sum(1 for i in after if i < 200)
        assert all(i < 200 for i in after[:k]) and all(i >= 200 for i in after[k:])


def test_eviction_clears_exactly_the_mapped_bits(orc):
    rng = np.random.default_rng(3)
    P = orc.OraclePool(1, 64, 64, 1, 128)
    r = P.open()
    bits = np.where(rng.random(500) < 0.5, 2, 4).astype(np.uint8)
    assert P.append(np.full(500, r), bits) == orc.OK
    ev = rng.choice(500, 40, replace=False)
    assert P.evict(np.full(40, r), ev) == orc.OK
    ex = P.export(r, content=False)
    dead = sum(int(f) - bin(int(l)).count("1") for f, l in zip(ex["fill"], ex["live"]))
    assert dead == 40
    assert P.evict(np.full(40, r), ev) == orc.OK                      # idempotent
    assert P.export(r, content=False)["live"].tolist() == ex["live"].tolist()
    assert P.evict([r], [500]) == orc.INVALID


def test_oom_and_invalid_leave_state_unchanged(orc):
    P = orc.OraclePool(1, 2, 3, 2, 8)
    r = P.open()
    assert P.append(np.full(40, r), np.full(40, 4, np.uint8)) == orc.OK   # 2 INT4 pages
    before = P.export(r, content=False)
    assert P.append(np.full(64, r), np.full(64, 4, np.uint8)) == orc.OOM  # needs 2 more, 1 free
    assert P.append(np.full(1, r), np.full(1, 5, np.uint8)) == orc.INVALID
    assert P.append(np.full(1, r), np.full(1, 3, np.uint8)) == orc.OOM       # no INT3 pages in this pool
    assert P.append(np.full(1, 1), np.full(1, 4, np.uint8)) == orc.INVALID  # request 1 not open
    after = P.export(r, content=False)
    for key in before:
        assert np.array_equal(before[key], after[key])
    k = np.zeros((1, 1, 128), np.uint16)
    k[0, 0, 5] = 0x7F80                                                     # +inf in bf16
    assert P.append([r], [4], k, k) == orc.RANGE


def test_repack_requantizes_int4_values_per_channel_k_per_token_v(orc):
    """The INT2 page built at the 32nd INT2 token equals INT2 quantization of the
    staging page's INT4-dequantized values: K per channel over the 32 tokens,
    V per token over 32-channel groups.  Live bits carry over."""
    P = orc.OraclePool(2, 4, 4, 1, 8, sel_heads=[1])
    r = P.open()
    k, v = _kv(32, 2, 0)
    assert P.append(np.full(31, r), np.full(31, 2, np.uint8), k[:31, 1:2], v[:31, 1:2]) == orc.OK
    assert P.evict([r], [4]) == orc.OK
    st = P.export(r)
    assert P.append([r], [2], k[31:, 1:2], v[31:, 1:2]) == orc.OK
    # staging content for slot 31 = INT4 quantization of token 31, taken from a
    # fresh request holding just that token as INT4
    P2 = orc.OraclePool(2, 4, 4, 1, 8, sel_heads=[1])
    r2 = P2.open()
    assert P2.append([r2], [4], k[31:, 1:2], v[31:, 1:2]) == orc.OK
    last = P2.export(r2)
    Ks, Vs = dequant_page(st["kc"][0, 0], st["vc"][0, 0], st["km"][0, 0], st["vm"][0, 0], False)
    K1, V1 = dequant_page(last["kc"][0, 0], last["vc"][0, 0], last["km"][0, 0], last["vm"][0, 0], False)
    Ks[31], Vs[31] = K1[0], V1[0]
    ex = P.export(r)
    assert ex["is_int2"].tolist() == [1] and ex["fill"].tolist() == [32]
    assert ex["live"][0] == 0xFFFFFFFF & ~(1 << 4)
    for c in range(128):
        codes, s, z = orc.quant_group(Ks[:, c], 2)
        assert np.array_equal(ex["kc"][0, 0, :, c], codes)
        assert ex["km"][0, 0, 2 * c] == s and ex["km"][0, 0, 2 * c + 1] == z
    for t in range(32):
        for g in range(4):
            codes, s, z = orc.quant_group(Vs[t, 32 * g:32 * g + 32], 2)
            assert np.array_equal(ex["vc"][0, 0, t, 32 * g:32 * g + 32], codes)
            assert ex["vm"][0, 0, (t * 4 + g) * 2] == s and ex["vm"][0, 0, (t * 4 + g) * 2 + 1] == z
