"""CUDA path vs oracle: codes, scale/zero and page tables bit-exact; attention
outputs within max-abs 1e-3 and relative-L2 1e-4 of the fp64 oracle."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_content, compare_tables

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 4242
SCALE = float(np.float32(1 / np.sqrt(128)))


IMPLS = [1, 2]   # KV_DECODE_SIMT, KV_DECODE_MMA


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


class Scenario:
    """Explicit requests (bit sequences, evictions) built on both sides with the
    same append call boundaries."""

    def __init__(self, kvq, hkv, hq, bits_list, chunk=64, evict=None, n2=None, n4=None, reorder=True,
                 impl=None, chan_mult=None):
        self.hkv, self.hq = hkv, hq
        n_req = len(bits_list)
        tot2 = sum(int((b == 2).sum()) for b in bits_list)
        tot4 = sum(int((b == 4).sum()) for b in bits_list)
        n2 = n2 or tot2 // 32 + 4
        n4 = n4 or tot4 // 32 + 2 * n_req + chunk // 32 + 8
        max_tab = max([int((b == 2).sum()) // 32 + int((b == 4).sum()) // 32 + 4 for b in bits_list] + [4])
        self.gpu = kvq.KVPool(hkv, n2, n4, n_req, max_tab)
        if impl is not None:
            self.gpu.set_decode_impl(impl)
        self.orc = oracle.OraclePool(hkv, n2, n4, n_req, max_tab)
        self.g_ids = [self.gpu.open() for _ in bits_list]
        self.o_ids = [self.orc.open() for _ in bits_list]
        self.cm = chan_mult
        dev = torch.device("cuda")
        cm_dev = None if chan_mult is None else torch.from_numpy(chan_mult).to(dev)
        for r, bits in enumerate(bits_list):
            n = bits.size
            for t0 in range(0, n, chunk):
                m = min(chunk, n - t0)
                kd = torch.empty((m, hkv, 128), dtype=torch.bfloat16, device=dev)
                vd = torch.empty((m, hkv, 128), dtype=torch.bfloat16, device=dev)
                kvsynth.fill_bf16_dev(kd.data_ptr(), m, hkv, 128, SEED, kvsynth.TENSOR_K, r, t0,
                                      cm_dev.data_ptr() if cm_dev is not None else 0)
                kvsynth.fill_bf16_dev(vd.data_ptr(), m, hkv, 128, SEED, kvsynth.TENSOR_V, r, t0)
                kh = kvsynth.fill_bf16_host(m, hkv, 128, SEED, kvsynth.TENSOR_K, r, t0, chan_mult=chan_mult)
                vh = kvsynth.fill_bf16_host(m, hkv, 128, SEED, kvsynth.TENSOR_V, r, t0)
                self.gpu.append(kd, vd, np.full(m, self.g_ids[r]), bits[t0:t0 + m])
                assert self.orc.append(np.full(m, self.o_ids[r]), bits[t0:t0 + m], kh, vh) == oracle.OK
        if evict:
            for r, pos in evict.items():
                self.gpu.evict(np.full(len(pos), self.g_ids[r]), pos)
                assert self.orc.evict(np.full(len(pos), self.o_ids[r]), pos) == oracle.OK
        if reorder:
            self.gpu.reorder(self.g_ids)
            assert self.orc.reorder(self.o_ids) == oracle.OK
        self.gpu.sync()

    def check_content(self):
        for g, o in zip(self.g_ids, self.o_ids):
            compare_content(self.gpu.export(g), self.orc.export(o), list(range(self.hkv)))

    def check_decode(self, step=0, what=""):
        B = len(self.g_ids)
        qd = torch.empty((B, self.hq, 128), dtype=torch.bfloat16, device="cuda")
        kvsynth.fill_bf16_dev(qd.data_ptr(), B, self.hq, 128, SEED, kvsynth.TENSOR_Q, step)
        qh = kvsynth.fill_bf16_host(B, self.hq, 128, SEED, kvsynth.TENSOR_Q, step)
        out = self.gpu.decode(qd, self.g_ids, SCALE)
        self.gpu.sync()
        ref = self.orc.decode(qh, self.o_ids, SCALE).reshape(B, self.hq, 128)
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        return assert_outputs_close(got, ref, what)


def _mixed(n, p2, seed):
    return np.where(np.random.default_rng(seed).random(n) < p2, 2, 4).astype(np.uint8)


def test_bulk_append_every_run(kvq):
    """Two one-request calls of 80 tokens laid out so that the second call
    completes the open tail page and opens a new one, completes the open
    staging page (repack), fills a 32-token group within the call (direct INT2)
    and leaves a partial staging page, with INT2 and INT4 tokens alternating
    (their page opens interleave).  Codes, tables and outputs against the
    oracle, which follows the per-token rules."""
    first = np.array([4, 2] * 30 + [4] * 20, np.uint8)      # 50 INT4 (tail 32 + 18), 30 INT2 (staging 30)
    second = np.array([2, 4] * 40, np.uint8)                 # 40 INT2: 2 + 32 + 6; 40 INT4: 14 + 26
    bits = [np.concatenate([first, second])]
    sc = Scenario(kvq, 2, 8, bits, chunk=80)
    sc.check_content()
    sc.check_decode(what="bulk runs")
    ex = sc.gpu.export(sc.g_ids[0], content=False)
    assert int(ex["is_int2"].sum()) == 2                     # the repacked staging page and the direct group
    assert int((ex["fill"] < 32).sum()) == 2                 # the partial INT4 tail and the partial staging page


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 63, 64, 65, 200])
@pytest.mark.parametrize("p2", [0.0, 0.5, 1.0])
def test_small_requests_codes_tables_outputs(kvq, n, p2, impl):
    bits = [_mixed(n, p2, n), _mixed(n + 7, p2, n + 1)]
    sc = Scenario(kvq, 2, 8, bits, chunk=48, impl=impl)
    sc.check_content()
    sc.check_decode(what=f"n={n} p2={p2} impl={impl}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hkv,hq", [(1, 1), (2, 4), (4, 12), (2, 16), (1, 7), (1, 2), (1, 3), (1, 5), (1, 6), (1, 8),
                                    (64, 64), (64, 512)])   # the largest kv head count: head 63 fills the ticket's field
def test_gqa_ratios(kvq, hkv, hq, impl):
    bits = [_mixed(300, 0.6, 1), _mixed(97, 0.3, 2), _mixed(1, 1.0, 3)]
    sc = Scenario(kvq, hkv, hq, bits, chunk=128, impl=impl)
    sc.check_content()
    sc.check_decode(what=f"hkv={hkv} hq={hq} impl={impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_outlier_channels_and_evictions(kvq, impl):
    cm = np.ones((2, 128), np.float32)
    cm[0, [3, 77, 90, 127]] = 20.0
    cm[1, [0, 31, 32, 64]] = 20.0
    bits = [_mixed(1000, 0.6, 5), _mixed(640, 0.8, 6)]
    rng = np.random.default_rng(7)
    ev = {0: rng.choice(1000, 50, replace=False), 1: rng.choice(640, 32, replace=False)}
    sc = Scenario(kvq, 2, 8, bits, chunk=256, evict=ev, chan_mult=cm, impl=impl)
    sc.check_content()
    sc.check_decode(what="outliers+evict")


@pytest.mark.parametrize("impl", IMPLS)
def test_all_dead_and_empty_requests(kvq, impl):
    bits = [_mixed(70, 0.5, 8), _mixed(40, 0.5, 9), np.zeros(0, np.uint8)]
    sc = Scenario(kvq, 2, 8, bits, evict={0: np.arange(70)}, impl=impl)
    out_ref = sc.check_decode(what="all-dead/empty")
    qd = torch.zeros((3, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = sc.gpu.decode(qd, sc.g_ids, SCALE).cpu().numpy()
    assert np.array_equal(out[0], np.zeros((8, 128), np.float32))
    assert np.array_equal(out[2], np.zeros((8, 128), np.float32))
    assert out_ref is not None


def test_unreordered_tables_and_interleaved_requests(kvq):
    """Tokens of three requests interleaved in one call; no reorder (mixed runs)."""
    rng = np.random.default_rng(10)
    n = 900
    req = rng.integers(0, 3, n)
    bits = np.where(rng.random(n) < 0.55, 2, 4).astype(np.uint8)
    hkv, hq = 2, 8
    gpu = kvq.KVPool(hkv, 64, 64, 3, 64)
    orc = oracle.OraclePool(hkv, 64, 64, 3, 64)
    g = [gpu.open() for _ in range(3)]
    o = [orc.open() for _ in range(3)]
    kd = torch.empty((n, hkv, 128), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    kvsynth.fill_bf16_dev(kd.data_ptr(), n, hkv, 128, SEED, kvsynth.TENSOR_K, 99)
    kvsynth.fill_bf16_dev(vd.data_ptr(), n, hkv, 128, SEED, kvsynth.TENSOR_V, 99)
    kh = kvsynth.fill_bf16_host(n, hkv, 128, SEED, kvsynth.TENSOR_K, 99)
    vh = kvsynth.fill_bf16_host(n, hkv, 128, SEED, kvsynth.TENSOR_V, 99)
    for a, b in ((0, 400), (400, 900)):
        gpu.append(kd[a:b], vd[a:b], np.array(g)[req[a:b]], bits[a:b])
        assert orc.append(np.array(o)[req[a:b]], bits[a:b], kh[a:b], vh[a:b]) == oracle.OK
    gpu.sync()
    for gi, oi in zip(g, o):
        compare_content(gpu.export(gi), orc.export(oi), [0, 1])
    qd = torch.empty((3, hq, 128), dtype=torch.bfloat16, device="cuda")
    kvsynth.fill_bf16_dev(qd.data_ptr(), 3, hq, 128, SEED, kvsynth.TENSOR_Q, 0)
    qh = kvsynth.fill_bf16_host(3, hq, 128, SEED, kvsynth.TENSOR_Q, 0)
    out = gpu.decode(qd, g, SCALE).cpu().numpy()
    assert_outputs_close(out, orc.decode(qh, o, SCALE).reshape(3, hq, 128), "interleaved")


def test_close_reuse_and_oom_leave_state(kvq):
    hkv = 1
    gpu = kvq.KVPool(hkv, 4, 4, 2, 16)
    orc = oracle.OraclePool(hkv, 4, 4, 2, 16)
    a, oa = gpu.open(), orc.open()
    k = torch.zeros((100, hkv, 128), dtype=torch.bfloat16, device="cuda")
    bits = np.full(100, 4, np.uint8)
    gpu.append(k, k, np.full(100, a), bits)
    assert orc.append(np.full(100, oa), bits) == oracle.OK
    before = gpu.export(a, content=False)
    with pytest.raises(kvq.KVError) as e:
        gpu.append(k[:64], k[:64], np.full(64, a), bits[:64])
    assert e.value.status == kvq.KV_ERR_OOM
    assert orc.append(np.full(64, oa), bits[:64]) == oracle.OOM
    compare_tables(gpu.export(a, content=False), before)
    gpu.close_request(a)
    orc.close_request(oa)
    b, ob = gpu.open(), orc.open()
    gpu.append(k[:33], k[:33], np.full(33, b), np.full(33, 2, np.uint8))
    assert orc.append(np.full(33, ob), np.full(33, 2, np.uint8)) == oracle.OK
    compare_tables(gpu.export(b, content=False), orc.export(ob, content=False))


def test_table_capacity_limit_leaves_state(kvq):
    """A request's table holds at most max_pages_per_request entries: a call
    that would pass it returns KV_ERR_OOM on both sides (bulk call of one
    request, and tokens of two requests interleaved) and changes nothing; a
    call that fits then proceeds as on the oracle."""
    hkv, cap = 2, 4
    gpu = kvq.KVPool(hkv, 32, 32, 2, cap)
    orc = oracle.OraclePool(hkv, 32, 32, 2, cap)
    g = [gpu.open() for _ in range(2)]
    o = [orc.open() for _ in range(2)]
    kh = kvsynth.fill_bf16_host(300, hkv, 128, SEED, kvsynth.TENSOR_K, 5)
    vh = kvsynth.fill_bf16_host(300, hkv, 128, SEED, kvsynth.TENSOR_V, 5)
    kd, vd = torch.from_numpy(kh.view(np.int16)).cuda().view(torch.bfloat16), \
        torch.from_numpy(vh.view(np.int16)).cuda().view(torch.bfloat16)
    bits = np.full(300, 4, np.uint8)
    gpu.append(kd[:100], vd[:100], np.full(100, g[0]), bits[:100])            # 4 INT4 pages: the table is full
    assert orc.append(np.full(100, o[0]), bits[:100], kh[:100], vh[:100]) == oracle.OK
    gpu.sync()
    before = [gpu.export(x, content=False) for x in g]
    with pytest.raises(kvq.KVError) as e:                                      # bulk: one request, 200 tokens
        gpu.append(kd[100:300], vd[100:300], np.full(200, g[0]), bits[100:300])
    assert e.value.status == kvq.KV_ERR_OOM
    assert orc.append(np.full(200, o[0]), bits[100:300], kh[100:300], vh[100:300]) == oracle.OOM
    req = np.where(np.arange(200) % 2 == 0, 0, 1)                              # per token: interleaved requests
    with pytest.raises(kvq.KVError) as e:
        gpu.append(kd[100:300], vd[100:300], np.array(g)[req], bits[100:300])
    assert e.value.status == kvq.KV_ERR_OOM
    assert orc.append(np.array(o)[req], bits[100:300], kh[100:300], vh[100:300]) == oracle.OOM
    gpu.sync()
    for x, b in zip(g, before):
        compare_tables(gpu.export(x, content=False), b)
    gpu.append(kd[100:128], vd[100:128], np.full(28, g[0]), bits[100:128])    # fills the last page's 28 free slots
    assert orc.append(np.full(28, o[0]), bits[100:128], kh[100:128], vh[100:128]) == oracle.OK
    gpu.sync()
    for x, y in zip(g, o):
        compare_content(gpu.export(x), orc.export(y), [0, 1])


def test_range_error_reported_by_sync(kvq):
    gpu = kvq.KVPool(1, 4, 4, 1, 8)
    a = gpu.open()
    k = torch.zeros((3, 1, 128), dtype=torch.bfloat16, device="cuda")
    k[1, 0, 5] = float("inf")
    gpu.append(k, torch.zeros_like(k), [a] * 3, [4] * 3)
    with pytest.raises(kvq.KVError) as e:
        gpu.sync()
    assert e.value.status == kvq.KV_ERR_RANGE
    gpu.sync()   # cleared


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("p2", [0.0, 1.0, 0.6])
def test_split_counts_do_not_change_results(kvq, p2, impl):
    """Long single request: many splits per unit vs the oracle."""
    bits = [_mixed(20000, p2, 11)]
    sc = Scenario(kvq, 1, 8, bits, chunk=4096, impl=impl)
    sc.check_decode(what=f"long p2={p2}")
    assert sc.gpu.last_decode_stats()["n_splits"] > 1


@pytest.mark.parametrize("impl", IMPLS)
def test_plan_reuse_across_growth(kvq, impl):
    """Decode, grow the tables (an empty request gains its first pages, others
    grow by a few pages, then by many), decode again: every call must scan
    every page, whether the decode plan was reused or rebuilt."""
    hkv, hq = 2, 8
    gpu = kvq.KVPool(hkv, 64, 64, 3, 64)
    orc = oracle.OraclePool(hkv, 64, 64, 3, 64)
    g = [gpu.open() for _ in range(3)]
    o = [orc.open() for _ in range(3)]
    gpu.set_decode_impl(impl)
    lens = [300, 40, 0]
    pos = [0, 0, 0]

    def grow(r, n, stream):
        if n == 0:
            return
        bits = _mixed(n, 0.5, 100 + stream)
        kd = torch.empty((n, hkv, 128), dtype=torch.bfloat16, device="cuda")
        vd = torch.empty_like(kd)
        kvsynth.fill_bf16_dev(kd.data_ptr(), n, hkv, 128, SEED, kvsynth.TENSOR_K, r, pos[r])
        kvsynth.fill_bf16_dev(vd.data_ptr(), n, hkv, 128, SEED, kvsynth.TENSOR_V, r, pos[r])
        kh = kvsynth.fill_bf16_host(n, hkv, 128, SEED, kvsynth.TENSOR_K, r, pos[r])
        vh = kvsynth.fill_bf16_host(n, hkv, 128, SEED, kvsynth.TENSOR_V, r, pos[r])
        gpu.append(kd, vd, np.full(n, g[r]), bits)
        assert orc.append(np.full(n, o[r]), bits, kh, vh) == oracle.OK
        pos[r] += n

    def check(step, what):
        qd = torch.empty((3, hq, 128), dtype=torch.bfloat16, device="cuda")
        kvsynth.fill_bf16_dev(qd.data_ptr(), 3, hq, 128, SEED, kvsynth.TENSOR_Q, step)
        qh = kvsynth.fill_bf16_host(3, hq, 128, SEED, kvsynth.TENSOR_Q, step)
        out = gpu.decode(qd, g, SCALE).cpu().numpy()
        gpu.sync()
        assert_outputs_close(out, orc.decode(qh, o, SCALE).reshape(3, hq, 128), what)

    for r in range(3):
        grow(r, lens[r], r)
    gpu.reorder(g)
    assert orc.reorder(o) == oracle.OK
    check(0, "initial (request 2 empty)")
    for step, add in enumerate(([5, 33, 70], [1, 1, 1], [3, 0, 2], [400, 200, 300]), start=1):
        for r in range(3):
            grow(r, add[r], 10 * step + r)
        gpu.reorder(g)
        assert orc.reorder(o) == oracle.OK
        check(step, f"after growth {add}")


def test_decode_timing_samples_every_nth_call(kvq):
    bits = [_mixed(200, 0.5, 21), _mixed(90, 0.5, 22)]
    sc = Scenario(kvq, 2, 8, bits)
    qd = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    n0, _, _ = sc.gpu.decode_timing(True, every=3)
    for _ in range(7):
        sc.gpu.decode(qd, sc.g_ids, SCALE)
    n, scan_ms, dec_ms = sc.gpu.decode_timing(False)
    assert n == 3                                   # calls 1, 4 and 7
    assert 0.0 < scan_ms <= dec_ms
    sc.gpu.decode_timing(True)                      # restart: counts from zero, every call
    sc.gpu.decode(qd, sc.g_ids, SCALE)
    n, _, _ = sc.gpu.decode_timing(False)
    assert n == 1
    assert kvq.load_library().kv_decode_timing(sc.gpu.handle, -1, None, None, None) == kvq.KV_ERR_INVALID_ARG
