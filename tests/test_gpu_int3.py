"""CUDA path vs oracle with INT3 pages beside INT2 and INT4 (TriAxialKV,
limitations and outlook: INT3 as a further width; K and V per token in
32-channel groups, codes 0..7, stored as a 2-bit and a 1-bit plane).
Tables, codes and binary16 scale/zero bits must equal the oracle's; outputs
of both scans within max-abs 1e-3 and relative-L2 1e-4 of the fp64 oracle."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_content, compare_tables
from test_gpu_parity import SCALE, SEED

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

IMPLS = [1, 2]   # KV_DECODE_SIMT, KV_DECODE_MMA


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _dev(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).cuda()


def _mixed3(n, seed, p=(0.4, 0.35, 0.25)):
    return np.random.default_rng(seed).choice(np.array([2, 3, 4], np.uint8), n, p=list(p))


class Pools:
    """One GPU pool and its oracle twin with INT3 pages, fed the same calls."""

    def __init__(self, kvq, hkv, hq, n_req, n2, n3, n4, max_tab, impl=None, nf=0):
        self.kvq, self.hkv, self.hq = kvq, hkv, hq
        self.nf_first = n2 + n4 + n3 if nf else None   # FP4 ids follow the INT3 ids
        self.gpu = kvq.KVPool(hkv, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        if impl is not None:
            self.gpu.set_decode_impl(impl)
        self.orc = oracle.OraclePool(hkv, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        self.g = [self.gpu.open() for _ in range(n_req)]
        self.o = [self.orc.open() for _ in range(n_req)]
        self.n = [0] * n_req

    def append(self, rs, bits, stream0=0):
        """One call: token q goes to request rs[q] with width bits[q]."""
        rs = np.asarray(rs)
        n = rs.size
        k = np.zeros((n, self.hkv, 128), np.uint16)
        v = np.zeros_like(k)
        for q, r in enumerate(rs):
            k[q] = kvsynth.fill_bf16_host(1, self.hkv, 128, SEED, kvsynth.TENSOR_K, stream0 + int(r), self.n[r])[0]
            v[q] = kvsynth.fill_bf16_host(1, self.hkv, 128, SEED, kvsynth.TENSOR_V, stream0 + int(r), self.n[r])[0]
            self.n[r] += 1
        self.gpu.append(_dev(k), _dev(v), np.array([self.g[r] for r in rs], np.int32), bits)
        assert self.orc.append(np.array([self.o[r] for r in rs], np.int32), bits, k, v) == oracle.OK

    def append_run(self, r, bits, stream0=0):
        self.append(np.full(np.asarray(bits).size, r), bits, stream0)

    def check_content(self):
        self.gpu.sync()
        for g, o in zip(self.g, self.o):
            compare_content(self.gpu.export(g), self.orc.export(o), list(range(self.hkv)))

    def check_decode(self, step, what):
        B = len(self.g)
        qh = kvsynth.fill_bf16_host(B, self.hq, 128, SEED, kvsynth.TENSOR_Q, step)
        out = self.gpu.decode(_dev(qh), self.g, SCALE)
        self.gpu.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        ref = self.orc.decode(qh, self.o, SCALE).reshape(B, self.hq, 128)
        return assert_outputs_close(got, ref, what)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hkv,hq", [(2, 8), (1, 8), (2, 16), (4, 4), (1, 3)])
def test_mixed_widths_prefill_reorder_decode(kvq, impl, hkv, hq):
    """Two requests of mixed 2/3/4-bit tokens in 100-token calls (fresh INT3
    pages, INT3 tails growing across calls), reorder, decode; then decode
    steps with one token per request per call."""
    P = Pools(kvq, hkv, hq, 2, 40, 40, 60, 64, impl=impl)
    bits = [_mixed3(700, 1), _mixed3(333, 2)]
    for r in range(2):
        for a in range(0, bits[r].size, 100):
            P.append_run(r, bits[r][a:a + 100])
    P.check_content()
    P.gpu.reorder(P.g)
    assert P.orc.reorder(P.o) == oracle.OK
    P.gpu.sync()
    for g, o in zip(P.g, P.o):
        compare_tables(P.gpu.export(g, content=False), P.orc.export(o, content=False))
    P.check_decode(0, f"mixed widths impl={impl} g={hq // hkv}")
    for step in range(1, 40):
        P.append([0, 1], _mixed3(2, 100 + step))
        P.gpu.reorder(P.g)
        assert P.orc.reorder(P.o) == oracle.OK
        if step % 13 == 0:
            P.check_decode(step, f"decode step {step}")
    P.check_content()
    P.check_decode(99, "after 39 steps")


@pytest.mark.parametrize("impl", IMPLS)
def test_int3_only_and_interleaved_requests(kvq, impl):
    """An all-INT3 request, and a call whose tokens alternate requests and
    widths token by token (three tails per request open in one call)."""
    P = Pools(kvq, 2, 8, 3, 16, 40, 40, 40, impl=impl)
    P.append_run(0, np.full(300, 3, np.uint8))
    rs = np.tile([1, 2], 250)
    P.append(rs, _mixed3(500, 5, p=(0.3, 0.4, 0.3)))
    P.check_content()
    P.check_decode(0, f"int3 only + interleaved impl={impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_int3_with_evictions_exclusion_and_drop(kvq, impl):
    """Evictions (sentinel dead slots), per-head exclusion (the scan variant
    with exclusion words) and dropping dead pages, INT3 pages among them."""
    rng = np.random.default_rng(8)
    P = Pools(kvq, 2, 8, 2, 40, 40, 60, 64, impl=impl)
    for r, n in enumerate([640, 400]):
        b = _mixed3(n, 10 + r)
        for a in range(0, n, 128):
            P.append_run(r, b[a:a + 128])
    for r in range(2):
        pos = np.sort(rng.choice(P.n[r], P.n[r] // 4, replace=False))
        P.gpu.evict(np.full(pos.size, P.g[r]), pos)
        assert P.orc.evict(np.full(pos.size, P.o[r]), pos) == oracle.OK
        cut = np.arange(P.n[r] // 2)
        P.gpu.evict_head(np.full(cut.size, P.g[r]), cut, np.zeros(cut.size, np.int32))
        assert P.orc.evict_head(np.full(cut.size, P.o[r]), cut, np.zeros(cut.size, np.int32)) == oracle.OK
        lead = np.arange(160)
        P.gpu.evict(np.full(lead.size, P.g[r]), lead)
        assert P.orc.evict(np.full(lead.size, P.o[r]), lead) == oracle.OK
    P.gpu.reorder(P.g)
    assert P.orc.reorder(P.o) == oracle.OK
    P.check_decode(0, f"evict + exclusion impl={impl}")
    n_before = [P.gpu.info(g)[0] for g in P.g]
    P.gpu.drop_dead_pages(P.g)
    assert P.orc.drop_dead_pages(P.o) == oracle.OK
    P.gpu.sync()
    assert sum(P.gpu.info(g)[0] for g in P.g) < sum(n_before)
    P.check_content()
    P.check_decode(1, f"after drop impl={impl}")
    # freed INT3 ids are taken again lowest first
    P.append_run(0, np.full(70, 3, np.uint8))
    P.check_content()
    P.check_decode(2, f"after refill impl={impl}")


def test_larger_mixed_workload_sampled(kvq):
    """4 requests x 3000-6000 tokens (INT2 0.45 / INT3 0.35 / INT4 0.2) in
    1024-token calls, g = 8, tensor-core scan: tables bit-exact, outputs of
    two sampled units per request against the oracle's selected heads."""
    hkv, hq, n_req = 4, 32, 4
    ns = [3000, 4500, 6000, 3333]
    bits = [_mixed3(n, 40 + r, p=(0.45, 0.35, 0.2)) for r, n in enumerate(ns)]
    n2 = sum(int((b == 2).sum()) for b in bits) // 32 + 8
    n3 = sum(int((b == 3).sum()) for b in bits) // 32 + 8
    n4 = sum(int((b == 4).sum()) for b in bits) // 32 + 64
    gpu = kvq.KVPool(hkv, n2, n4, n_req, 256, n_int3_pages=n3)
    sel = [1, 3]
    orc = oracle.OraclePool(hkv, n2, n4, n_req, 256, sel_heads=sel, n_int3_pages=n3)
    g = [gpu.open() for _ in ns]
    o = [orc.open() for _ in ns]
    for r, n in enumerate(ns):
        for a in range(0, n, 1024):
            m = min(1024, n - a)
            k = kvsynth.fill_bf16_host(m, hkv, 128, SEED, kvsynth.TENSOR_K, 60 + r, a)
            v = kvsynth.fill_bf16_host(m, hkv, 128, SEED, kvsynth.TENSOR_V, 60 + r, a)
            gpu.append(_dev(k), _dev(v), np.full(m, g[r], np.int32), bits[r][a:a + m])
            assert orc.append(np.full(m, o[r]), bits[r][a:a + m], k[:, sel], v[:, sel]) == oracle.OK
    gpu.reorder(g)
    assert orc.reorder(o) == oracle.OK
    qh = kvsynth.fill_bf16_host(n_req, hq, 128, SEED, kvsynth.TENSOR_Q, 3)
    out = gpu.decode(_dev(qh), g, SCALE)
    gpu.sync()
    for r in range(n_req):
        ge, oe = gpu.export(g[r], content=False), orc.export(o[r], content=False)
        compare_tables(ge, oe)
    gq = hq // hkv
    pairs = np.array([(b, h * gq + j) for b in range(n_req) for h in sel for j in range(gq)], np.int32)
    ref = orc.decode(qh, o, SCALE, pairs=pairs)
    got = out.cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    assert_outputs_close(got, ref, "3000-6000 tokens, g = 8")


def test_int3_errors(kvq):
    """Width 3 in a pool without INT3 pages is out of pages; width 5 is
    invalid.  A grouped decode over a pool with INT3 pages and one without
    gives each pool's own decode."""
    gpu = kvq.KVPool(1, 4, 4, 1, 8)
    r = gpu.open()
    k = _dev(kvsynth.fill_bf16_host(1, 1, 128, SEED, kvsynth.TENSOR_K, 0))
    with pytest.raises(kvq.KVError) as e:
        gpu.append(k, k, [r], [3])
    assert e.value.status == kvq.KV_ERR_OOM
    with pytest.raises(kvq.KVError) as e:
        gpu.append(k, k, [r], [5])
    assert e.value.status == kvq.KV_ERR_INVALID_ARG
    assert gpu.info(r) == (0, 0)
    a = kvq.KVPool(1, 4, 4, 1, 8, n_int3_pages=4)
    b = kvq.KVPool(1, 4, 4, 1, 8)
    ra, rb = a.open(), b.open()
    a.append(k, k, [ra], [3])
    b.append(k, k, [rb], [4])
    q = _dev(kvsynth.fill_bf16_host(1, 2, 128, SEED, kvsynth.TENSOR_Q, 0))
    out = kvq.KVPool.decode_groups([a, b], q, np.array([[ra], [rb]], np.int32), SCALE)
    oa = a.decode(q[:, :1].contiguous(), [ra], SCALE)
    ob = b.decode(q[:, 1:].contiguous(), [rb], SCALE)
    a.sync()
    got = out.cpu().numpy()
    assert_outputs_close(got[:, :1], oa.cpu().numpy(), "grouped INT3 pool")
    assert_outputs_close(got[:, 1:], ob.cpu().numpy(), "grouped INT4 pool")


def test_config2_full_size_three_width_allocation(kvq):
    """The 32K-token batch-8 workload at full size with the three-width
    allocation (kv_alloc_bits3 over the same budget; `bench.py --config 2
    --alloc3` builds the same pool): the widths equal the oracle's
    allocation, every table bit-exact, sampled units' codes and outputs
    within the tolerance, over 3 decode steps."""
    from harness import OracleWorkload
    from mixed_precision_kv_gb300.workload import GPUWorkload, int3_pages, pool_size
    steps = 3
    w = kvsynth.make_workload(2, steps=steps)
    gw = GPUWorkload(w, steps=steps, three_widths=True)
    n3 = int3_pages(w, gw.bits, steps)
    assert n3 > 0
    sel, reqs = [0, 5], [2, 7]
    ow = OracleWorkload(w, pool_size(w, gw.bits, gw.chunk, gw.steps), gw.chunk, sel_heads=sel, content_reqs=reqs,
                        n_int3_pages=n3, three_widths=True)
    for a, b in zip(gw.bits, ow.bits):
        assert np.array_equal(a, b)
    assert any((b == 3).any() for b in gw.bits)
    gw.prefill()
    ow.prefill()
    gw.evict()
    ow.evict()
    gw.reorder()
    ow.reorder()
    gw.pool.sync()
    g = w.g

    def check(step, content):
        out = gw.decode(gw.q(step)).cpu().numpy()
        gw.pool.sync()
        for r in range(len(gw.rids)):
            compare_tables(gw.pool.export(gw.rids[r], content=False), ow.P.export(ow.rids[r], content=False))
        if content:
            for r in reqs:
                compare_content(gw.pool.export(gw.rids[r]), ow.P.export(ow.rids[r]), sel)
        pairs = np.array([(b, h * g + x) for b in reqs for h in sel for x in range(g)], np.int32)
        ref = ow.decode(ow.q(step), pairs=pairs)
        got = np.stack([out[b, hq] for b, hq in pairs])
        assert np.isfinite(got).all()
        assert_outputs_close(got, ref, f"32K batch 8 three-width allocation, step {step}")

    check(0, True)
    for step in range(1, steps + 1):
        k, v, _, bits = gw.step_inputs()
        gw.append_step(k, v, np.array(gw.rids, np.int32), bits)
        ow.append_step()
        gw.reorder()
        ow.reorder()
        check(step, step == steps)
