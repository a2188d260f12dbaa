"""Oracle pins for INT3 pages, the further width the TriAxialKV page's
limitations and outlook section names beside INT2 and INT4 (reading: K and V
per token in 32-channel groups as INT4, codes 0..7; INT3 page ids after the
INT2 and INT4 ranges; a request's INT3 tokens fill its own INT3 tail;
the phase-1 reorder sorts tables stably by width).

What fixes the results here: closed forms of ids, fills and table order;
attention recomputed by an independent numpy restatement from the export
(np_ref.attention_from_export); an all-INT3 request equals plain softmax
attention over an independently written per-token INT3 quantization; a
split-merge and page-order invariance."""
import numpy as np
import pytest

import kvsynth
from np_ref import attention_from_export, quant_tokens_np

SCALE = float(np.float32(1 / np.sqrt(128)))


def _kv(n, hkv, stream, seed=5, tok0=0):
    return (kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_K, stream, tok0),
            kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_V, stream, tok0))


def _q(B, Hq, seed=9):
    return kvsynth.fill_bf16_host(B, Hq, 128, seed, kvsynth.TENSOR_Q, 0)


def test_routing_ids_and_width_sorted_reorder(orc):
    P = orc.OraclePool(2, 4, 8, 1, 16, n_int3_pages=8)
    r = P.open()
    bits = np.array([3] * 40 + [4] * 10 + [2] * 32, np.uint8)
    k, v = _kv(bits.size, 2, 0)
    assert P.append(np.full(bits.size, r), bits, k, v) == orc.OK
    ex = P.export(r, content=False)
    # INT4 ids [4, 12), INT3 ids [12, 20): INT3 pages 12 (32 tokens) and 13
    # (8); the INT4 tail 4 (10) and the staging page 5, repacked into INT2
    # id 0 and freed
    assert ex["ids"].tolist() == [12, 13, 4, 0]
    assert ex["fill"].tolist() == [32, 8, 10, 32]
    assert ex["is_int2"].tolist() == [0, 0, 0, 1]
    assert P.reorder([r]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [0, 12, 13, 4]
    # the next staging page takes the freed INT4 id 5; INT3 tokens continue in page 13
    k2, v2 = _kv(3, 2, 0, tok0=bits.size)
    assert P.append(np.full(3, r), np.array([2, 3, 4], np.uint8), k2, v2) == orc.OK
    ex = P.export(r, content=False)
    assert ex["ids"].tolist() == [0, 12, 13, 4, 5]
    assert ex["fill"].tolist() == [32, 32, 9, 11, 1]


def test_reorder_is_a_stable_sort_by_width(orc):
    P = orc.OraclePool(1, 8, 16, 1, 32, n_int3_pages=16)
    r = P.open()
    # one call per run so that the pages open in this order: 4, 3, 2 (via staging), 4, 3, 2
    runs = [(4, 32), (3, 32), (2, 32), (4, 32), (3, 32), (2, 32)]
    t0 = 0
    for b, n in runs:
        k, v = _kv(n, 1, 1, tok0=t0)
        assert P.append(np.full(n, r), np.full(n, b, np.uint8), k, v) == orc.OK
        t0 += n
    before = P.export(r, content=False)["ids"].tolist()
    # INT4 ids [8, 24), INT3 ids [24, 40); each staging page (9, then 10) is
    # repacked into INT2 (0, 1) and its id freed for the next INT4 page
    assert before == [8, 24, 0, 9, 25, 1]
    assert P.reorder([r]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [0, 1, 24, 25, 8, 9]


def _mixed3(n, rng):
    return rng.choice(np.array([2, 3, 4], np.uint8), n, p=[0.4, 0.35, 0.25])


@pytest.mark.parametrize("n", [1, 31, 33, 100])
def test_decode_brute_force_with_int3_pages(orc, n):
    rng = np.random.default_rng(n)
    P = orc.OraclePool(2, 64, 64, 2, 64, n_int3_pages=64)
    rids, q = [], _q(2, 8)
    for i, m in enumerate([n, 170 - n]):
        r = P.open()
        k, v = _kv(m, 2, i)
        assert P.append(np.full(m, r), _mixed3(m, rng), k, v) == orc.OK
        ev = rng.choice(m, m // 5, replace=False)
        assert P.evict(np.full(ev.size, r), ev) == orc.OK
        rids.append(r)
    out = P.decode(q, rids, SCALE)
    for b, r in enumerate(rids):
        ex = P.export(r)
        i3 = (ex["ids"] >= 128) & (ex["ids"] < 192)                # INT3 ids [n2 + n4, n2 + n4 + n3)
        assert i3.any() and int(ex["kc"][i3].max()) <= 7 and int(ex["vc"][i3].max()) <= 7
        for hq in range(8):
            ref = attention_from_export(ex, hq // 4, kvsynth.bf16_to_f32(q[b, hq]), SCALE)
            np.testing.assert_allclose(out[b * 8 + hq], ref, rtol=1e-12, atol=1e-13)
    base = out
    for s in (2, 5, 64):
        np.testing.assert_allclose(P.decode(q, rids, SCALE, n_splits=s), base, rtol=1e-12, atol=1e-14)
    assert P.reorder(rids) == orc.OK
    np.testing.assert_allclose(P.decode(q, rids, SCALE), base, rtol=1e-12, atol=1e-14)


def test_int3_codes_stay_below_eight(orc):
    P = orc.OraclePool(2, 4, 4, 1, 16, n_int3_pages=8)
    r = P.open()
    k, v = _kv(96, 2, 3)
    assert P.append(np.full(96, r), np.full(96, 3, np.uint8), k, v) == orc.OK
    ex = P.export(r)
    assert ex["ids"].tolist() == [8, 9, 10]
    assert int(ex["kc"].max()) == 7 and int(ex["vc"].max()) == 7


def test_all_int3_equals_uniform_per_token_int3_attention(orc):
    n = 250
    P = orc.OraclePool(2, 4, 4, 1, 16, n_int3_pages=16)
    r = P.open()
    k, v = _kv(n, 2, 4)
    assert P.append(np.full(n, r), np.full(n, 3, np.uint8), k, v) == orc.OK
    q = _q(1, 8)
    out = P.decode(q, [r], SCALE)
    for hq in range(8):
        kv = hq // 4
        K = quant_tokens_np(kvsynth.bf16_to_f32(k[:, kv]), 3).astype(np.float64)
        V = quant_tokens_np(kvsynth.bf16_to_f32(v[:, kv]), 3).astype(np.float64)
        lg = SCALE * (K @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out[hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-13)


def test_int3_lies_between_int2_and_int4_in_error(orc):
    """Per-token INT3 error against the bf16 values sits between INT4's and
    the coarser 2-bit per-token grid's on the same rows (a sanity property
    of a narrower grid, checked on 400 tokens)."""
    k, _ = _kv(400, 1, 6)
    x = kvsynth.bf16_to_f32(k[:, 0])
    e = {b: float(np.abs(quant_tokens_np(x, b) - x).mean()) for b in (2, 3, 4)}
    assert e[4] < e[3] < e[2]
    P = orc.OraclePool(1, 4, 16, 1, 32, n_int3_pages=16)
    r = P.open()
    assert P.append(np.full(400, r), np.full(400, 3, np.uint8), k, k) == orc.OK
    ex = P.export(r)
    got = np.concatenate([
        (ex["kc"][i, 0].astype(np.float64)
         * np.repeat(ex["km"][i, 0].reshape(32, 4, 2)[:, :, 0].view(np.float16).astype(np.float64), 32, 1)
         + np.repeat(ex["km"][i, 0].reshape(32, 4, 2)[:, :, 1].view(np.float16).astype(np.float64), 32, 1)
         )[:int(ex["fill"][i])] for i in range(ex["ids"].size)])
    np.testing.assert_allclose(got.astype(np.float32), quant_tokens_np(x, 3), rtol=0, atol=0)


def test_int3_oom_invalid_drop_and_close(orc):
    P = orc.OraclePool(1, 2, 2, 2, 8, n_int3_pages=2)
    r = P.open()
    k, v = _kv(65, 1, 7)
    assert P.append(np.full(65, r), np.full(65, 3, np.uint8), k, v) == orc.OOM    # 3 INT3 pages needed, 2 exist
    assert P.info(r) == (0, 0)
    assert P.append(np.full(1, r), np.array([5], np.uint8), k[:1], v[:1]) == orc.INVALID
    assert P.append(np.full(64, r), np.full(64, 3, np.uint8), k[:64], v[:64]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [4, 5]                  # INT3 ids [4, 6)
    assert P.evict(np.full(32, r), np.arange(32)) == orc.OK
    assert P.drop_dead_pages([r]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [5]
    s = P.open()
    assert P.append(np.full(1, s), np.array([3], np.uint8), k[:1], v[:1]) == orc.OK
    assert P.export(s, content=False)["ids"].tolist() == [4]                     # the dropped id, lowest free
    P.close_request(r)
    assert P.append(np.full(33, s), np.full(33, 3, np.uint8), k[:33], v[:33]) == orc.OK
    assert P.export(s, content=False)["ids"].tolist() == [4, 5]
