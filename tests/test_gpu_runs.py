"""Calls made of per-request runs (one chunk of each of several requests, the
shape of a batched chunked prefill): codes, scale/zero, page tables and
positions bit-exact against the oracle, which routes every token by the
per-token rules; outputs within max-abs 1e-3 and relative-L2 1e-4."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_content

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 5151
SCALE = float(np.float32(1 / np.sqrt(128)))
HKV, HQ = 2, 8


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


class Pools:
    """A GPU pool and an oracle pool fed the same calls; request r's tokens are
    its positions 0, 1, ... in the order they are appended."""

    def __init__(self, kvq, bits_list, n2, n4, max_tab):
        self.bits = bits_list
        self.gpu = kvq.KVPool(HKV, n2, n4, len(bits_list), max_tab)
        self.orc = oracle.OraclePool(HKV, n2, n4, len(bits_list), max_tab)
        self.g = [self.gpu.open() for _ in bits_list]
        self.o = [self.orc.open() for _ in bits_list]
        self.pos = [0] * len(bits_list)

    def rows(self, r, t0, m):
        kd = torch.empty((m, HKV, 128), dtype=torch.bfloat16, device="cuda")
        vd = torch.empty_like(kd)
        kvsynth.fill_bf16_dev(kd.data_ptr(), m, HKV, 128, SEED, kvsynth.TENSOR_K, r, t0)
        kvsynth.fill_bf16_dev(vd.data_ptr(), m, HKV, 128, SEED, kvsynth.TENSOR_V, r, t0)
        kh = kvsynth.fill_bf16_host(m, HKV, 128, SEED, kvsynth.TENSOR_K, r, t0)
        vh = kvsynth.fill_bf16_host(m, HKV, 128, SEED, kvsynth.TENSOR_V, r, t0)
        return kd, vd, kh, vh

    def call(self, runs, expect=None):
        """One append call: runs = [(request, n tokens), ...] in call order."""
        kd, vd, kh, vh, gr, orq, bb = [], [], [], [], [], [], []
        for r, m in runs:
            t0 = self.pos[r]
            a, b, c, d = self.rows(r, t0, m)
            kd.append(a); vd.append(b); kh.append(c); vh.append(d)
            gr.append(np.full(m, self.g[r], np.int32))
            orq.append(np.full(m, self.o[r], np.int32))
            bb.append(self.bits[r][t0:t0 + m])
        bits = np.ascontiguousarray(np.concatenate(bb))
        if expect is not None:
            with pytest.raises(kvq_error()) as ei:
                self.gpu.append(torch.cat(kd), torch.cat(vd), np.concatenate(gr), bits)
            assert ei.value.status == expect
            assert self.orc.append(np.concatenate(orq), bits, np.concatenate(kh), np.concatenate(vh)) == expect
            return
        self.gpu.append(torch.cat(kd), torch.cat(vd), np.concatenate(gr), bits)
        assert self.orc.append(np.concatenate(orq), bits, np.concatenate(kh), np.concatenate(vh)) == oracle.OK
        for r, m in runs:
            self.pos[r] += m

    def check(self, what):
        self.gpu.sync()
        for g, o in zip(self.g, self.o):
            ge, oe = self.gpu.export(g), self.orc.export(o)
            compare_content(ge, oe, list(range(HKV)))
        self.gpu.reorder(self.g)
        assert self.orc.reorder(self.o) == oracle.OK
        B = len(self.g)
        qd = torch.empty((B, HQ, 128), dtype=torch.bfloat16, device="cuda")
        kvsynth.fill_bf16_dev(qd.data_ptr(), B, HQ, 128, SEED, kvsynth.TENSOR_Q, 0)
        qh = kvsynth.fill_bf16_host(B, HQ, 128, SEED, kvsynth.TENSOR_Q, 0)
        out = self.gpu.decode(qd, self.g, SCALE).cpu().numpy()
        assert np.isfinite(out).all()
        assert_outputs_close(out, self.orc.decode(qh, self.o, SCALE).reshape(B, HQ, 128), what)


def kvq_error():
    import mixed_precision_kv_gb300 as m
    return m.KVError


def _bits(n, p2, seed):
    return np.where(np.random.default_rng(seed).random(n) < p2, 2, 4).astype(np.uint8)


def test_runs_of_several_requests(kvq):
    """Four requests appended in calls that carry one chunk of each (runs of
    33 to 300 tokens): tail and staging pages carried across calls, repacks,
    direct INT2 groups and partial pages in every run.  Then a call with a
    run shorter than a page and a call with a request in two runs (both
    routed token by token), evictions by position, and a decode."""
    bits = [_bits(2000, p2, 10 + r) for r, p2 in enumerate([0.0, 0.35, 0.6, 1.0])]
    P = Pools(kvq, bits, n2=120, n4=200, max_tab=80)
    P.call([(0, 100), (1, 33), (2, 300), (3, 64)])
    P.check("runs, first call")
    P.call([(2, 77), (0, 40), (3, 95), (1, 250)])
    P.call([(1, 128), (3, 32), (0, 200), (2, 61)])
    P.check("runs, three calls")
    P.call([(0, 31), (1, 90), (2, 45)])            # a run shorter than a page
    P.call([(3, 40), (2, 50), (3, 40)])            # request 3 in two runs
    P.call([(2, 150), (1, 70), (0, 99), (3, 36)])
    for r in range(4):
        pos = np.random.default_rng(70 + r).choice(P.pos[r], 25, replace=False).astype(np.int64)
        P.gpu.evict(np.full(pos.size, P.g[r]), pos)
        assert P.orc.evict(np.full(pos.size, P.o[r]), pos) == oracle.OK
    P.check("runs, after the fallback calls and evictions")


def test_runs_out_of_pages_change_nothing(kvq):
    """A call whose runs need more INT4 pages than are free: KV_ERR_OOM on both
    sides and the pool as before (tables, codes, the next call's result)."""
    bits = [_bits(1000, 0.5, 30 + r) for r in range(3)]
    P = Pools(kvq, bits, n2=40, n4=14, max_tab=64)
    P.call([(0, 64), (1, 64), (2, 64)])
    before = [P.gpu.export(g) for g in P.g]
    P.call([(0, 200), (1, 200), (2, 200)], expect=oracle.OOM)
    P.gpu.sync()
    for b, g in zip(before, P.g):
        a = P.gpu.export(g)
        for key in ("ids", "is_int2", "fill", "live"):
            assert np.array_equal(a[key], b[key]), key
    P.call([(2, 40), (0, 40)])
    P.check("runs after an OOM")


def test_interleaved_prefill_full_size(kvq):
    """The 32K-token batch-8 prompts appended in calls that carry 4096 tokens
    of every request: every table bit-exact, codes and scale/zero of two kv
    heads of every request, and their decode outputs, against the oracle."""
    from harness import OracleWorkload
    from mixed_precision_kv_gb300.workload import GPUWorkload, pool_size
    w = kvsynth.make_workload(2)
    per, heads = 4096, [1, 6]
    chunk = per * len(w.requests)
    gw = GPUWorkload(w, chunk=chunk)
    ow = OracleWorkload(w, pool_size(w, gw.bits, chunk, gw.steps), chunk, sel_heads=heads)
    for a, b in zip(gw.bits, ow.bits):
        assert np.array_equal(a, b)
    n = max(s.n_prefill for s in w.requests)
    for t0 in range(0, n, per):
        gk, gv, ok_, ov, gr, orq, bb = [], [], [], [], [], [], []
        for r, spec in enumerate(w.requests):
            m = min(per, spec.n_prefill - t0)
            if m <= 0:
                continue
            k, v = gw.kv_rows(r, t0, m)
            kh, vh = ow.kv_rows(r, t0, m)
            gk.append(k); gv.append(v); ok_.append(kh); ov.append(vh)
            gr.append(np.full(m, gw.rids[r], np.int32))
            orq.append(np.full(m, ow.rids[r], np.int32))
            bb.append(gw.bits[r][t0:t0 + m])
        bits = np.ascontiguousarray(np.concatenate(bb))
        gw.pool.append(torch.cat(gk), torch.cat(gv), np.concatenate(gr), bits)
        assert ow.P.append(np.concatenate(orq), bits, np.concatenate(ok_), np.concatenate(ov)) == oracle.OK
    gw.reorder()
    ow.reorder()
    gw.pool.sync()
    for r in range(len(w.requests)):
        compare_content(gw.pool.export(gw.rids[r]), ow.P.export(ow.rids[r]), heads)
    g = w.g
    pairs = [(b, h * g + j) for b in range(len(w.requests)) for h in heads for j in range(g)]
    out = gw.decode(gw.q(0)).cpu().numpy()
    gw.pool.sync()
    ref = ow.decode(ow.q(0), pairs=np.array(pairs, np.int32))
    got = np.stack([out[b, h] for b, h in pairs])
    assert_outputs_close(got, ref, "interleaved prefill, full size")
