"""Oracle pins for dropping dead pages and for head groups held in pools of
their own (Tangram, method steps 6-7: head groups keep different amounts of
context, each holding only its own pages; IntentKV, method 2: surviving pages
do not move).

What fixes the results here:
  - closed forms of the table after a drop and of the ids the next pages take
    (lowest free id, R5);
  - a dead slot contributes exactly 0 to the fp64 softmax (e^(-1e4 - m)
    underflows), so dropping pages whose slots are all dead leaves every
    output bit-identical;
  - per-(page, head) quantization does not look at other heads, so a head
    group's own pool, fed the same tokens, holds the shared pool's blocks for
    its heads, and after it evicts and drops what its budget excludes its
    outputs equal the shared pool's with those positions excluded for the
    group's heads only."""
import numpy as np
import pytest

import kvsynth

SEED = 77
SCALE = float(np.float32(1 / np.sqrt(128)))


def _rows(n, H, stream, tok0=0):
    k = kvsynth.fill_bf16_host(n, H, 128, SEED, kvsynth.TENSOR_K, stream, tok0)
    v = kvsynth.fill_bf16_host(n, H, 128, SEED, kvsynth.TENSOR_V, stream, tok0)
    return k, v


def _pool(orc, H, n2=32, n4=64, reqs=2, max_tab=64):
    P = orc.OraclePool(H, n2, n4, reqs, max_tab)
    return P, [P.open() for _ in range(reqs)]


def test_drop_keeps_order_and_frees_lowest_ids(orc):
    P, (r, _) = _pool(orc, 2, n2=4, n4=16)
    k, v = _rows(160, 2, 0)
    assert P.append(np.full(160, r), np.full(160, 4, np.uint8), k, v) == orc.OK
    ids = P.export(r, content=False)["ids"].tolist()
    assert ids == [4, 5, 6, 7, 8]                       # INT4 ids start after the 4 INT2 ids
    dead = np.concatenate([np.arange(32, 64), np.arange(96, 128)])
    assert P.evict(np.full(dead.size, r), dead) == orc.OK
    assert P.drop_dead_pages([r]) == orc.OK
    ex = P.export(r, content=False)
    assert ex["ids"].tolist() == [4, 6, 8]              # order kept
    assert ex["live"].tolist() == [0xFFFFFFFF] * 3
    # the tail page (8) is full: the next INT4 token opens a page with the lowest free id, 5
    k2, v2 = _rows(1, 2, 0, 160)
    assert P.append([r], [4], k2, v2) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [4, 6, 8, 5]


def test_drop_keeps_partial_and_partly_live_pages(orc):
    P, (r, _) = _pool(orc, 2, n2=4, n4=16)
    k, v = _rows(112, 2, 1)
    assert P.append(np.full(112, r), np.full(112, 4, np.uint8), k, v) == orc.OK   # pages 4, 5, 6 full; 7 holds 16
    # page 4: one slot still live; page 5: dead for head 0 only; page 6: dead for both heads; page 7: all dead, partial
    assert P.evict(np.full(31, r), np.arange(31)) == orc.OK
    assert P.evict_head(np.full(32, r), np.arange(32, 64), np.zeros(32, np.int32)) == orc.OK
    pos = np.arange(64, 96)
    assert P.evict_head(np.full(64, r), np.concatenate([pos, pos]), np.repeat([0, 1], 32).astype(np.int32)) == orc.OK
    assert P.evict(np.full(16, r), np.arange(96, 112)) == orc.OK
    assert P.drop_dead_pages([r]) == orc.OK
    assert P.export(r, content=False)["ids"].tolist() == [4, 5, 7]


def test_drop_leaves_every_output_bit_identical(orc):
    rng = np.random.default_rng(5)
    H, hq = 2, 8
    P, rids = _pool(orc, H)
    for j, r in enumerate(rids):
        n = 300 + 97 * j
        bits = np.where(rng.random(n) < 0.6, 2, 4).astype(np.uint8)
        k, v = _rows(n, H, 10 + j)
        assert P.append(np.full(n, r), bits, k, v) == orc.OK
    assert P.reorder(rids) == orc.OK
    for r in rids:
        # scattered slots evicted, and the first 96 positions (whole pages among them)
        n_tok = P.info(r)[1]
        pos = np.sort(rng.choice(n_tok, n_tok // 2, replace=False))
        assert P.evict(np.full(pos.size, r), pos) == orc.OK
        assert P.evict(np.full(96, r), np.arange(96)) == orc.OK
    q = kvsynth.fill_bf16_host(2, hq, 128, SEED, kvsynth.TENSOR_Q, 0)
    before = P.decode(q, rids, SCALE)
    n_before = [P.info(r)[0] for r in rids]
    assert P.drop_dead_pages(rids) == orc.OK
    n_after = [P.info(r)[0] for r in rids]
    assert sum(n_after) < sum(n_before)
    after = P.decode(q, rids, SCALE)
    assert np.array_equal(before, after)


def test_evict_after_drop_changes_nothing(orc):
    P, (r, _) = _pool(orc, 2, n2=4, n4=16)
    k, v = _rows(96, 2, 3)
    assert P.append(np.full(96, r), np.full(96, 4, np.uint8), k, v) == orc.OK
    assert P.evict(np.full(32, r), np.arange(32)) == orc.OK
    assert P.drop_dead_pages([r]) == orc.OK
    ex0 = P.export(r)
    q = kvsynth.fill_bf16_host(1, 4, 128, SEED, kvsynth.TENSOR_Q, 1)
    o0 = P.decode(q, [r], SCALE)
    assert P.evict(np.full(4, r), np.array([0, 5, 31, 40])) == orc.OK                 # 0..31 were on the dropped page
    assert P.evict_head(np.full(2, r), np.array([3, 7]), np.array([0, 1], np.int32)) == orc.OK
    ex1 = P.export(r)
    assert int(ex1["live"][0]) == int(ex0["live"][0]) & ~(1 << (40 - 32))              # only position 40 changed
    o1 = P.decode(q, [r], SCALE)
    assert not np.array_equal(o0, o1)
    P2, (r2, _) = _pool(orc, 2, n2=4, n4=16)
    assert P2.append(np.full(96, r2), np.full(96, 4, np.uint8), k, v) == orc.OK
    assert P2.evict(np.full(33, r2), np.concatenate([np.arange(32), [40]])) == orc.OK
    assert np.array_equal(o1, P2.decode(q, [r2], SCALE))


@pytest.mark.parametrize("keep_frac", [0.0, 0.4, 0.77])
def test_head_group_pools_equal_shared_pool_with_exclusion(orc, keep_frac):
    """Kv heads 0-1 form group 0 (keeps everything), heads 2-3 group 1 (keeps
    the most recent keep_frac of each request).  Shared pool S: per-head
    exclusion of group 1's dropped positions.  Group pools A (heads 0-1) and B
    (heads 2-3): the same tokens, bits and call boundaries; B evicts those
    positions and drops its dead pages; B0 is B before the drop.  Outputs
    (g = 2) of A and B must equal S's in fp64.  B0 must hold S's tables (ids
    included: allocation does not depend on heads) and S's blocks for heads
    2-3; B must be B0 without its full, wholly dead pages, in order."""
    rng = np.random.default_rng(9)
    H, g = 4, 2
    hq = H * g
    S, srid = _pool(orc, H, n2=48, n4=96, reqs=3)
    A, arid = _pool(orc, 2, n2=48, n4=96, reqs=3)
    B, brid = _pool(orc, 2, n2=48, n4=96, reqs=3)
    B0, b0rid = _pool(orc, 2, n2=48, n4=96, reqs=3)
    for j in range(3):
        n = 400 + 150 * j
        bits = np.where(rng.random(n) < 0.6, 2, 4).astype(np.uint8)
        for t0 in range(0, n, 128):
            m = min(128, n - t0)
            k, v = _rows(m, H, 20 + j, t0)
            assert S.append(np.full(m, srid[j]), bits[t0:t0 + m], k, v) == orc.OK
            assert A.append(np.full(m, arid[j]), bits[t0:t0 + m], k[:, :2], v[:, :2]) == orc.OK
            for P, r in ((B, brid), (B0, b0rid)):
                assert P.append(np.full(m, r[j]), bits[t0:t0 + m], k[:, 2:], v[:, 2:]) == orc.OK
        c = n - int(round(keep_frac * n))
        pos = np.arange(c, dtype=np.int64)
        assert S.evict_head(np.full(2 * c, srid[j]), np.concatenate([pos, pos]),
                            np.repeat([2, 3], c).astype(np.int32)) == orc.OK
        for P, r in ((B, brid), (B0, b0rid)):
            assert P.evict(np.full(c, r[j]), pos) == orc.OK
    for P, r in ((S, srid), (A, arid), (B, brid), (B0, b0rid)):
        assert P.reorder(r) == orc.OK
    assert B.drop_dead_pages(brid) == orc.OK
    q = kvsynth.fill_bf16_host(3, hq, 128, SEED, kvsynth.TENSOR_Q, 2)
    shared = S.decode(q, srid, SCALE).reshape(3, hq, 128)
    grouped = np.concatenate([A.decode(q[:, :4], arid, SCALE).reshape(3, 4, 128),
                              B.decode(q[:, 4:], brid, SCALE).reshape(3, 4, 128)], axis=1)
    assert np.array_equal(shared, grouped)
    dropped = 0
    for j in range(3):
        se, b0, be = S.export(srid[j]), B0.export(b0rid[j]), B.export(brid[j])
        assert np.array_equal(se["ids"], b0["ids"]) and np.array_equal(se["fill"], b0["fill"])
        assert np.array_equal(se["is_int2"], b0["is_int2"])
        for key in ("kc", "vc", "km", "vm"):
            assert np.array_equal(se[key][:, 2:], b0[key])
        kept = [i for i in range(b0["ids"].size) if not (b0["fill"][i] == 32 and b0["live"][i] == 0)]
        dropped += b0["ids"].size - len(kept)
        assert be["ids"].tolist() == b0["ids"][kept].tolist()
        for key in ("is_int2", "fill", "live", "kc", "vc", "km", "vm"):
            assert np.array_equal(be[key], b0[key][kept])
    assert dropped > 0
