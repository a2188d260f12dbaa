"""The five decode workloads, CUDA path vs oracle.

Small instances are compared in full (every code, scale/zero, table entry and
output).  Full-size instances are compared on every request's page table
(bit-exact) and on whole requests, all kv heads, whose codes and outputs the
oracle computes (workload 2: every request).
"""
import numpy as np
import pytest

import kvsynth
from harness import OracleWorkload, assert_outputs_close, compare_content, compare_tables

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _pair(w, chunk, steps=None, sel_heads=None, content_reqs=None, impl=None):
    from mixed_precision_kv_gb300.workload import GPUWorkload, pool_size
    gw = GPUWorkload(w, chunk=chunk, steps=steps)
    if impl is not None:
        gw.pool.set_decode_impl(impl)
    ow = OracleWorkload(w, pool_size(w, gw.bits, chunk, gw.steps), chunk, sel_heads=sel_heads,
                        content_reqs=content_reqs)
    for a, b in zip(gw.bits, ow.bits):
        assert np.array_equal(a, b)
    return gw, ow


def _build(gw, ow):
    gw.prefill()
    ow.prefill()
    gw.evict()
    ow.evict()
    gw.reorder()
    ow.reorder()
    gw.pool.sync()


def _check_all(gw, ow, reqs=None, content=True):
    for r in (range(len(gw.rids)) if reqs is None else reqs):
        ge = gw.pool.export(gw.rids[r], content=content)
        oe = ow.P.export(ow.rids[r], content=content)
        if content:
            compare_content(ge, oe, ow.sel)
        else:
            compare_tables(ge, oe)


def _decode_check(gw, ow, step, pairs=None, what=""):
    out = gw.decode(gw.q(step)).cpu().numpy()
    gw.pool.sync()
    q = ow.q(step)
    if pairs is None:
        ref = ow.decode(q).reshape(out.shape)
        got = out
    else:
        ref = ow.decode(q, pairs=pairs)
        got = np.stack([out[b, h] for b, h in pairs])
    assert np.isfinite(got).all()
    return assert_outputs_close(got, ref, what)


@pytest.mark.parametrize("impl", [1, 2])
def test_config1_full(kvq, impl):
    w = kvsynth.make_workload(1)
    gw, ow = _pair(w, chunk=512, impl=impl)
    _build(gw, ow)
    _check_all(gw, ow)
    frac2 = (gw.bits[0][:2048] == 2).mean()
    assert 0.5 <= frac2 <= 0.8
    _decode_check(gw, ow, 0, what="config 1")


@pytest.mark.parametrize("cfg,kw", [
    (2, dict(n_req=3, ctx=4000)),
    (3, dict(n_req=2, ctx=6000)),
    (4, dict(n_req=6, ctx_range=(300, 6000))),
])
def test_configs_small_full_compare(kvq, cfg, kw):
    w = kvsynth.make_workload(cfg, **kw)
    gw, ow = _pair(w, chunk=1024)
    _build(gw, ow)
    _check_all(gw, ow)
    _decode_check(gw, ow, 0, what=f"config {cfg} small")


def test_config5_loop_small(kvq):
    """Append one token per request per step, repack at 32 qualifying tokens,
    reorder, decode: tables every step, codes and outputs along the way."""
    w = kvsynth.make_workload(5, n_req=6, ctx_range=(100, 1500), steps=70)
    gw, ow = _pair(w, chunk=512)
    _build(gw, ow)
    repacks = 0
    for step in range(w.steps):
        k, v, rids, bits = gw.step_inputs()
        gw.append_step(k, v, rids, bits)
        ow.append_step()
        gw.reorder()
        ow.reorder()
        _check_all(gw, ow, content=(step % 10 == 9))
        _decode_check(gw, ow, step, what=f"config 5 step {step}")
        repacks += int((bits == 2).sum())
    assert repacks > 32


def _sampled(w, rng, n_units, n_heads=2):
    """Sample (request, kv head) units; return the sampled requests, heads and (b, q head) pairs."""
    reqs = sorted(set(rng.choice(len(w.requests), n_units, replace=False).tolist()))
    heads = sorted(set(rng.choice(w.num_kv_heads, n_heads, replace=False).tolist()))
    g = w.g
    pairs = [(b, h * g + j) for b in reqs for h in heads for j in range(g)]
    return reqs, heads, pairs


@pytest.mark.parametrize("cfg,n_req", [(2, 8), (3, 4)])
def test_configs_full_size_sampled(kvq, cfg, n_req):
    """Every table; codes, scale/zero and outputs of n_req requests with all
    their kv heads: config 2 every output (8 x 32 q heads), config 3 256 of
    the 1024 (request, q head) outputs."""
    w = kvsynth.make_workload(cfg)
    rng = np.random.default_rng(cfg)
    reqs, heads, pairs = _sampled(w, rng, n_req, n_heads=w.num_kv_heads)
    gw, ow = _pair(w, chunk=16384, sel_heads=heads, content_reqs=reqs)
    _build(gw, ow)
    _check_all(gw, ow, content=False)                 # every table, bit-exact
    _check_all(gw, ow, reqs=reqs, content=True)       # sampled codes and scale/zero
    q = ow.q(0)
    out = gw.decode(gw.q(0)).cpu().numpy()
    ref = ow.decode(q, pairs=np.array(pairs, np.int32), n_threads=0)
    got = np.stack([out[b, h] for b, h in pairs])
    assert_outputs_close(got, ref, f"config {cfg} full size, sampled")


def test_config4_full_size_sampled(kvq):
    """Every table; codes, scale/zero and outputs of the shortest, the longest
    and six seeded requests, with all their kv heads."""
    w = kvsynth.make_workload(4)
    rng = np.random.default_rng(44)
    lens = np.array([r.n_prefill for r in w.requests])
    ends = {int(np.argmin(lens)), int(np.argmax(lens))}
    rest = [b for b in range(len(w.requests)) if b not in ends]
    reqs = sorted(ends | set(rng.choice(rest, 6, replace=False).tolist()))
    heads = list(range(w.num_kv_heads))
    pairs = [(b, h * w.g + j) for b in reqs for h in heads for j in range(w.g)]
    gw, ow = _pair(w, chunk=16384, sel_heads=heads, content_reqs=reqs)
    _build(gw, ow)
    _check_all(gw, ow, content=False)
    _check_all(gw, ow, reqs=reqs, content=True)
    out = gw.decode(gw.q(0)).cpu().numpy()
    ref = ow.decode(ow.q(0), pairs=np.array(pairs, np.int32))
    got = np.stack([out[b, h] for b, h in pairs])
    assert_outputs_close(got, ref, "config 4 full size, sampled")


def test_config2_full_size_segments_and_budgets(kvq):
    """The 32K-token batch-8 workload with per-head budgets (kv head h keeps the
    most recent (h + 1)/8 of each prompt; whole pages are skipped) and
    full-precision segments (5 % vertical lines per kv head, a 128-token
    window), both as the bench sets them up; sampled units against the oracle."""
    w = kvsynth.make_workload(2)
    rng = np.random.default_rng(22)
    reqs, heads, pairs = _sampled(w, rng, 1)
    gw, ow = _pair(w, chunk=16384, sel_heads=heads, content_reqs=reqs)
    _build(gw, ow)
    H = w.num_kv_heads
    for r, spec in enumerate(w.requests):
        n = spec.n_prefill
        cuts = [n - int(round(n * (h + 1) / H)) for h in range(H)]
        pos = np.concatenate([np.arange(c, dtype=np.int64) for c in cuts])
        hh = np.concatenate([np.full(c, h, np.int32) for h, c in enumerate(cuts)])
        gw.pool.evict_head(np.full(pos.size, gw.rids[r], np.int32), pos, hh)
        if r in reqs:
            assert ow.P.evict_head(np.full(pos.size, ow.rids[r]), pos, hh) == 0
    window, rho = 128, 0.05
    gw.freeze_segments(rho=rho, window=window, staging=128)
    for r in reqs:
        n = w.requests[r].n_prefill
        pre = n - window
        nv = int(rho * pre)
        score = np.random.default_rng([w.seed, 77, r]).random((H, pre))
        pos = [np.sort(np.argpartition(score[h], pre - nv)[pre - nv:]) for h in range(H)]
        o = ow.rids[r]
        assert ow.P.evict_head(np.full(nv * H, o), np.concatenate(pos), np.repeat(np.arange(H), nv)) == 0
        assert ow.P.evict(np.full(window, o), np.arange(pre, n)) == 0
        k_all, v_all = ow.kv_rows(r, 0, n)
        kf = np.stack([k_all[pos[h], j] for j, h in enumerate(ow.sel)], axis=1)
        vf = np.stack([v_all[pos[h], j] for j, h in enumerate(ow.sel)], axis=1)
        assert ow.P.fp_append(o, kf, vf) == 0
        assert ow.P.fp_append(o, k_all[pre:n], v_all[pre:n]) == 0
    gw.reorder()
    ow.reorder()
    gw.pool.sync()
    out = gw.decode(gw.q(0)).cpu().numpy()
    gw.pool.sync()
    ref = ow.decode(ow.q(0), pairs=np.array(pairs, np.int32))
    got = np.stack([out[b, h] for b, h in pairs])
    assert np.isfinite(got).all()
    assert_outputs_close(got, ref, "config 2 full size, budgets + segments, sampled")


def test_config5_full_size_every_step(kvq):
    """The serving loop at its stated size: 256 requests with contexts
    U[4K, 64K], 64 steps of append (one token per request into the INT4 tail
    or staging page) -> repack of every staging page that reaches 32 tokens ->
    INT2-first reorder -> decode.  Every step: all 256 page tables (ids,
    precision, fill, live masks) bit-exact against the oracle, which keeps
    codes only for the sampled requests and kv heads.  At steps 0, 31 and 63,
    at the first step after a repack in a sampled request, and every 8th step:
    codes and binary16 scale/zero of 8 sampled requests with all their kv
    heads, and their outputs within max-abs 1e-3 / relative-L2 1e-4 of the
    fp64 oracle."""
    w = kvsynth.make_workload(5)
    assert len(w.requests) == 256 and w.steps == 64
    rng = np.random.default_rng(55)
    # four requests whose staging page fills during the 64 steps (INT2 tokens
    # wait in it, 32 at a time), four drawn at random
    from harness import oracle_bits
    fills = []
    for r, spec in enumerate(w.requests):
        b = oracle_bits(w, r)
        n = spec.n_prefill
        fills.append(int((b[:n] == 2).sum()) % 32 + int((b[n:n + w.steps] == 2).sum()) >= 32)
    repacking = [r for r in range(len(w.requests)) if fills[r]]
    reqs = rng.choice(repacking, 4, replace=False).tolist()
    rest = [r for r in range(len(w.requests)) if r not in reqs]
    reqs = sorted(reqs + rng.choice(rest, 4, replace=False).tolist())
    heads = list(range(w.num_kv_heads))
    pairs = np.array([(b, h * w.g + j) for b in reqs for h in heads for j in range(w.g)], np.int32)
    gw, ow = _pair(w, chunk=16384, sel_heads=heads, content_reqs=reqs)
    _build(gw, ow)
    _check_all(gw, ow, content=False)

    def n_int2(r):
        return int(gw.pool.export(gw.rids[r], content=False)["is_int2"].sum())

    int2_before = {r: n_int2(r) for r in reqs}
    repack_seen = False
    checked, repacks = [], 0
    for step in range(w.steps):
        k, v, rids, bits = gw.step_inputs()
        gw.append_step(k, v, rids, bits)
        ow.append_step()
        gw.reorder()
        ow.reorder()
        _check_all(gw, ow, content=False)                     # all 256 tables, every step
        repacks += int((bits == 2).sum())
        after = {r: n_int2(r) for r in reqs}
        first_repack = not repack_seen and any(after[r] > int2_before[r] for r in reqs)
        repack_seen = repack_seen or first_repack
        if step in (0, 31, 63) or first_repack or step % 8 == 7:
            _check_all(gw, ow, reqs=reqs, content=True)
            _decode_check(gw, ow, step, pairs=pairs, what=f"config 5 full size, step {step}")
            checked.append(step)
        else:
            gw.decode(gw.q(step))
    gw.pool.sync()
    assert repack_seen, "no sampled request repacked a staging page in 64 steps"
    assert {0, 31, 63} <= set(checked)
