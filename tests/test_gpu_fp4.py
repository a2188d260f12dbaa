"""CUDA path vs oracle with FP4 (E2M1) pages beside INT2, INT3 and INT4
(TriAxialKV, limitations and outlook: non-uniform FP formats; HyQuant
background: s = max|X| / c_B).  Codes, binary16 scales and tables must equal
the oracle's; outputs of both scans within max-abs 1e-3 and relative-L2 1e-4
of the fp64 oracle."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_tables
from test_gpu_int3 import IMPLS, Pools, _dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FP4 = 0xF4


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _widths(n, seed, p=(0.35, 0.15, 0.2, 0.3)):
    return np.random.default_rng(seed).choice(np.array([2, 3, 4, FP4], np.uint8), n, p=list(p))


def _check_content(P):
    """Codes and scale bits of every written slot; FP4 pages export {s, 0}."""
    P.gpu.sync()
    for g, o in zip(P.g, P.o):
        ge, oe = P.gpu.export(g), P.orc.export(o)
        compare_tables(ge, oe)
        for i in range(oe["ids"].size):
            f = int(oe["fill"][i])
            for key in ("kc", "vc"):
                assert np.array_equal(ge[key][i, :, :f], oe[key][i, :, :f]), (i, key)
            if oe["is_int2"][i]:
                assert np.array_equal(ge["km"][i], oe["km"][i])
            else:
                assert np.array_equal(ge["km"][i, :, :8 * f], oe["km"][i, :, :8 * f]), (i, "km")
            assert np.array_equal(ge["vm"][i, :, :8 * f], oe["vm"][i, :, :8 * f]), (i, "vm")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hkv,hq", [(2, 8), (1, 8), (2, 16), (4, 4), (1, 3)])
def test_four_widths_prefill_reorder_decode(kvq, impl, hkv, hq):
    P = Pools(kvq, hkv, hq, 2, 40, 30, 50, 80, impl=impl, nf=40)
    bits = [_widths(700, 1), _widths(333, 2)]
    for r in range(2):
        for a in range(0, bits[r].size, 100):
            P.append_run(r, bits[r][a:a + 100])
    _check_content(P)
    P.gpu.reorder(P.g)
    assert P.orc.reorder(P.o) == oracle.OK
    P.gpu.sync()
    for g, o in zip(P.g, P.o):
        compare_tables(P.gpu.export(g, content=False), P.orc.export(o, content=False))
    P.check_decode(0, f"four widths impl={impl} g={hq // hkv}")
    for step in range(1, 30):
        P.append([0, 1], _widths(2, 100 + step))
        P.gpu.reorder(P.g)
        assert P.orc.reorder(P.o) == oracle.OK
        if step % 10 == 0:
            P.check_decode(step, f"decode step {step}")
    _check_content(P)
    P.check_decode(99, "after 29 steps")


@pytest.mark.parametrize("impl", IMPLS)
def test_fp4_only_edge_values_and_interleaving(kvq, impl):
    """An all-FP4 request whose groups hit every E2M1 midpoint and zero
    groups, and a call whose tokens alternate requests and widths."""
    P = Pools(kvq, 2, 8, 3, 16, 8, 40, 40, impl=impl, nf=40)
    n = 96
    k = np.zeros((n, 2, 128), np.float32)
    v = np.zeros((n, 2, 128), np.float32)
    mid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0])
    rng = np.random.default_rng(3)
    for t in range(n):
        if t % 7 == 3:
            continue                                         # an all-zero token: scale 0
        for h in range(2):
            scale = float(2.0 ** rng.integers(-6, 6))
            k[t, h] = np.tile(mid, 8)[rng.permutation(128)] * scale
            v[t, h] = rng.standard_normal(128) * scale
    kb = (k.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact in bf16
    vb = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    P.gpu.append(_dev(kb), _dev(vb), np.full(n, P.g[0], np.int32), np.full(n, FP4, np.uint8))
    assert P.orc.append(np.full(n, P.o[0]), np.full(n, FP4, np.uint8), kb, vb) == oracle.OK
    P.n[0] = n
    rs = np.tile([1, 2], 200)
    P.append(rs, _widths(400, 5))
    _check_content(P)
    P.check_decode(0, f"fp4 edges + interleaved impl={impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_fp4_evictions_exclusion_drop(kvq, impl):
    rng = np.random.default_rng(8)
    P = Pools(kvq, 2, 8, 2, 40, 20, 40, 80, impl=impl, nf=60)
    for r, n in enumerate([640, 400]):
        b = _widths(n, 10 + r, p=(0.3, 0.1, 0.2, 0.4))
        for a in range(0, n, 128):
            P.append_run(r, b[a:a + 128])
    for r in range(2):
        pos = np.sort(rng.choice(P.n[r], P.n[r] // 4, replace=False))
        P.gpu.evict(np.full(pos.size, P.g[r]), pos)
        assert P.orc.evict(np.full(pos.size, P.o[r]), pos) == oracle.OK
        cut = np.arange(P.n[r] // 2)
        P.gpu.evict_head(np.full(cut.size, P.g[r]), cut, np.ones(cut.size, np.int32))
        assert P.orc.evict_head(np.full(cut.size, P.o[r]), cut, np.ones(cut.size, np.int32)) == oracle.OK
        lead = np.arange(200)
        P.gpu.evict(np.full(lead.size, P.g[r]), lead)
        assert P.orc.evict(np.full(lead.size, P.o[r]), lead) == oracle.OK
    P.gpu.reorder(P.g)
    assert P.orc.reorder(P.o) == oracle.OK
    P.check_decode(0, f"fp4 evict + exclusion impl={impl}")
    P.gpu.drop_dead_pages(P.g)
    assert P.orc.drop_dead_pages(P.o) == oracle.OK
    _check_content(P)
    P.check_decode(1, f"fp4 after drop impl={impl}")
    P.append_run(1, np.full(70, FP4, np.uint8))
    _check_content(P)
    P.check_decode(2, f"fp4 after refill impl={impl}")


def test_fp4_errors(kvq):
    gpu = kvq.KVPool(1, 4, 4, 1, 8)
    r = gpu.open()
    k = _dev(kvsynth.fill_bf16_host(1, 1, 128, 4242, kvsynth.TENSOR_K, 0))
    with pytest.raises(kvq.KVError) as e:
        gpu.append(k, k, [r], [FP4])
    assert e.value.status == kvq.KV_ERR_OOM
    with pytest.raises(kvq.KVError) as e:
        gpu.append(k, k, [r], [0xF3])
    assert e.value.status == kvq.KV_ERR_INVALID_ARG


def test_config2_full_size_four_widths(kvq):
    """The 32K-token batch-8 workload at full size with 30 % of its INT4
    tokens made INT3 and 30 % FP4 (`bench.py --config 2 --int3-share 0.3
    --fp4-share 0.3` builds the same pool), then 4 decode steps: every table
    bit-exact, sampled units' codes and outputs against the oracle."""
    from harness import OracleWorkload, compare_content
    from mixed_precision_kv_gb300.workload import GPUWorkload, int3_pages, pool_size
    steps = 4
    w = kvsynth.make_workload(2, steps=steps)
    gw = GPUWorkload(w, steps=steps, int3_share=0.3, fp4_share=0.3)
    n3, nf = int3_pages(w, gw.bits, steps), int3_pages(w, gw.bits, steps, FP4)
    assert n3 > 0 and nf > 0
    sel, reqs = [2, 7], [1, 6]
    ow = OracleWorkload(w, pool_size(w, gw.bits, gw.chunk, gw.steps), gw.chunk, sel_heads=sel, content_reqs=reqs,
                        n_int3_pages=n3, n_fp4_pages=nf, int3_share=0.3, fp4_share=0.3)
    for a, b in zip(gw.bits, ow.bits):
        assert np.array_equal(a, b)
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
                ge, oe = gw.pool.export(gw.rids[r]), ow.P.export(ow.rids[r])
                compare_tables(ge, oe)
                for i in range(oe["ids"].size):
                    f = int(oe["fill"][i])
                    for j, h in enumerate(sel):
                        for key in ("kc", "vc"):
                            assert np.array_equal(ge[key][i, h, :f], oe[key][i, j, :f]), (r, i, h, key)
                        if not oe["is_int2"][i]:
                            assert np.array_equal(ge["km"][i, h, :8 * f], oe["km"][i, j, :8 * f]), (r, i, h)
                        assert np.array_equal(ge["vm"][i, h, :8 * f], oe["vm"][i, j, :8 * f]), (r, i, h)
        pairs = np.array([(b, h * g + x) for b in reqs for h in sel for x in range(g)], np.int32)
        ref = ow.decode(ow.q(step), pairs=pairs)
        got = np.stack([out[b, hq] for b, hq in pairs])
        assert np.isfinite(got).all()
        assert_outputs_close(got, ref, f"32K batch 8 four widths, step {step}")

    check(0, True)
    for step in range(1, steps + 1):
        k, v, _, bits = gw.step_inputs()
        gw.append_step(k, v, np.array(gw.rids, np.int32), bits)
        ow.append_step()
        gw.reorder()
        ow.reorder()
        check(step, step == steps)
