"""CUDA path vs oracle for dropping dead pages (kv_drop_dead_pages) and for
head groups held in pools of their own (kv_decode_attn_groups, Tangram:
head groups keep different amounts of context).

Tables, codes and scale/zero bits must match the oracle's group pools
exactly; outputs must be within max-abs 1e-3 and relative-L2 1e-4 of the
fp64 oracle's shared pool (every kv head in one pool, a group's left-out
positions excluded for the group's heads only), which the oracle's own pins
show equal to its group pools."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_content, compare_tables
from test_gpu_parity import SCALE, SEED, _mixed

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _dev(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).cuda()


def _rows(n, H, stream, tok0=0):
    k = kvsynth.fill_bf16_host(n, H, 128, SEED, kvsynth.TENSOR_K, stream, tok0)
    v = kvsynth.fill_bf16_host(n, H, 128, SEED, kvsynth.TENSOR_V, stream, tok0)
    return k, v


def _q(B, hq, step):
    qh = kvsynth.fill_bf16_host(B, hq, 128, SEED, kvsynth.TENSOR_Q, step)
    return qh, _dev(qh)


def _sizes(bits_list, chunk):
    n_req = len(bits_list)
    n2 = sum(int((b == 2).sum()) for b in bits_list) // 32 + 4
    n4 = sum(int((b == 4).sum()) for b in bits_list) // 32 + 2 * n_req + chunk // 32 + 8
    max_tab = max(len(b) // 32 + 8 for b in bits_list)
    return n2, n4, max_tab


def _extra(bits_list, width):
    """Pages for the tokens of one tail width (INT3 or FP4), 0 if none."""
    n = sum(int((b == width).sum()) for b in bits_list)
    return n // 32 + 2 * len(bits_list) + 4 if n else 0


class Groups:
    """A model with sum(groups) kv heads cut into consecutive head groups.
    GPU: one pool per group, fed the group's rows of every token, with the
    same call boundaries.  Oracle: the same group pools (tables and codes),
    and one shared pool S with every head (the output reference)."""

    def __init__(self, kvq, groups, hq, bits_list, chunk=128, stream0=0, extra=0):
        self.kvq = kvq
        self.groups = list(groups)
        self.lo = np.concatenate([[0], np.cumsum(groups)]).astype(int)
        self.hkv = int(self.lo[-1])
        self.hq = hq
        self.bits = [b.copy() for b in bits_list]
        self.chunk = chunk
        self.stream0 = stream0
        n2, n4, max_tab = _sizes(bits_list, chunk)
        n2, n4, max_tab = n2 + extra, n4 + extra, max_tab + extra
        n3, nf = _extra(bits_list, 3), _extra(bits_list, 0xF4)
        n3, nf = n3 + (extra if n3 else 0), nf + (extra if nf else 0)
        n_req = len(bits_list)
        self.gpu = [kvq.KVPool(h, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf) for h in groups]
        self.og = [oracle.OraclePool(h, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf) for h in groups]
        self.S = oracle.OraclePool(self.hkv, n2, n4, n_req, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        self.g_ids = [[p.open() for _ in bits_list] for p in self.gpu]
        self.o_ids = [[p.open() for _ in bits_list] for p in self.og]
        self.s_ids = [self.S.open() for _ in bits_list]
        self.n_tok = [0] * n_req
        for r, bits in enumerate(bits_list):
            self.append(r, bits)

    def append(self, r, bits):
        n = bits.size
        t_base = self.n_tok[r]
        for t0 in range(0, n, self.chunk):
            m = min(self.chunk, n - t0)
            k, v = _rows(m, self.hkv, self.stream0 + r, t_base + t0)
            b = bits[t0:t0 + m]
            assert self.S.append(np.full(m, self.s_ids[r]), b, k, v) == oracle.OK
            for j in range(len(self.groups)):
                lo, hi = self.lo[j], self.lo[j + 1]
                self.gpu[j].append(_dev(k[:, lo:hi]), _dev(v[:, lo:hi]), np.full(m, self.g_ids[j][r]), b)
                assert self.og[j].append(np.full(m, self.o_ids[j][r]), b, k[:, lo:hi], v[:, lo:hi]) == oracle.OK
        self.n_tok[r] += n

    def leave_out(self, j, r, pos):
        """Group j stops reading positions `pos` of request r: its pools evict
        them, S excludes them for the group's heads."""
        pos = np.asarray(pos, np.int64)
        if pos.size == 0:
            return
        self.gpu[j].evict(np.full(pos.size, self.g_ids[j][r]), pos)
        assert self.og[j].evict(np.full(pos.size, self.o_ids[j][r]), pos) == oracle.OK
        heads = np.repeat(np.arange(self.lo[j], self.lo[j + 1]), pos.size).astype(np.int32)
        assert self.S.evict_head(np.full(heads.size, self.s_ids[r]), np.tile(pos, self.groups[j]), heads) == oracle.OK

    def exclude_head(self, j, r, pos, local_head):
        """One kv head of group j stops reading `pos` (a per-head exclusion inside the group's pool)."""
        pos = np.asarray(pos, np.int64)
        hl = np.full(pos.size, local_head, np.int32)
        self.gpu[j].evict_head(np.full(pos.size, self.g_ids[j][r]), pos, hl)
        assert self.og[j].evict_head(np.full(pos.size, self.o_ids[j][r]), pos, hl) == oracle.OK
        hs = np.full(pos.size, self.lo[j] + local_head, np.int32)
        assert self.S.evict_head(np.full(pos.size, self.s_ids[r]), pos, hs) == oracle.OK

    def reorder(self):
        for j in range(len(self.groups)):
            self.gpu[j].reorder(self.g_ids[j])
            assert self.og[j].reorder(self.o_ids[j]) == oracle.OK
        assert self.S.reorder(self.s_ids) == oracle.OK

    def drop(self):
        for j in range(len(self.groups)):
            self.gpu[j].drop_dead_pages(self.g_ids[j])
            assert self.og[j].drop_dead_pages(self.o_ids[j]) == oracle.OK

    def sync(self):
        for p in self.gpu:
            p.sync()

    def check_tables(self, content=True):
        for j in range(len(self.groups)):
            for g, o in zip(self.g_ids[j], self.o_ids[j]):
                ge, oe = self.gpu[j].export(g, content=content), self.og[j].export(o, content=content)
                if content:
                    compare_content(ge, oe, list(range(self.groups[j])))
                else:
                    compare_tables(ge, oe)

    def decode(self, step, what):
        B = len(self.s_ids)
        qh, qd = _q(B, self.hq, step)
        out = self.kvq.KVPool.decode_groups(self.gpu, qd, np.array(self.g_ids, np.int32), SCALE)
        self.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        ref = self.S.decode(qh, self.s_ids, SCALE).reshape(B, self.hq, 128)
        assert_outputs_close(got, ref, what)
        return got


# ---- kv_drop_dead_pages ---------------------------------------------------

def test_drop_dead_pages_tables_codes_and_outputs(kvq):
    """Scattered evictions plus whole leading pages; drop; the tables, codes
    and ids match the oracle's, outputs of both scans match the oracle and
    are unchanged by the drop (within the tolerance: the split plan changes);
    new pages take the lowest freed ids; evicting a dropped position is a
    no-op on both sides."""
    rng = np.random.default_rng(11)
    bits = [_mixed(700, 0.6, 1), _mixed(450, 0.4, 2)]
    sc = Groups(kvq, [2], 8, bits, extra=12)
    for r, n in enumerate(sc.n_tok):
        pos = np.sort(rng.choice(n, n // 3, replace=False))
        sc.leave_out(0, r, np.union1d(pos, np.arange(160)))
    sc.reorder()
    sc.sync()
    before = sc.decode(0, "before drop")
    n_before = [sc.gpu[0].info(g)[0] for g in sc.g_ids[0]]
    sc.drop()
    sc.sync()
    n_after = [sc.gpu[0].info(g)[0] for g in sc.g_ids[0]]
    assert sum(n_after) < sum(n_before)
    assert n_after == [sc.og[0].info(o)[0] for o in sc.o_ids[0]]
    sc.check_tables()
    for impl in (1, 2):
        sc.gpu[0].set_decode_impl(impl)
        B = len(sc.s_ids)
        qh, qd = _q(B, sc.hq, 0)
        got = sc.gpu[0].decode(qd, sc.g_ids[0], SCALE)
        sc.gpu[0].sync()
        ref = sc.og[0].decode(qh, sc.o_ids[0], SCALE).reshape(B, sc.hq, 128)
        assert_outputs_close(got.cpu().numpy(), ref, f"after drop impl={impl}")
        assert_outputs_close(got.cpu().numpy(), before, f"drop leaves outputs impl={impl}")
    # new tokens: the lowest freed ids first, on both sides
    for r in range(2):
        sc.append(r, _mixed(130, 0.5, 20 + r))
    sc.sync()
    sc.check_tables()
    # positions on dropped pages: evicting them again changes nothing
    sc.gpu[0].evict(np.full(3, sc.g_ids[0][0]), np.array([0, 31, 100]))
    assert sc.og[0].evict(np.full(3, sc.o_ids[0][0]), np.array([0, 31, 100])) == oracle.OK
    sc.sync()
    sc.check_tables(content=False)
    sc.decode(1, "after drop and appends")


def test_drop_keeps_partial_pages_and_heads_still_reading(kvq):
    """A page dead for one kv head only, a partial all-dead page and the
    staging page stay; only full pages dead for every head leave."""
    bits = [np.array([4] * 112 + [2] * 20, np.uint8)]
    sc = Groups(kvq, [2], 8, bits, chunk=132)
    g = sc.g_ids[0][0]
    sc.leave_out(0, 0, np.arange(31))                                  # page 0: one slot live
    sc.exclude_head(0, 0, np.arange(32, 64), 0)                        # page 1: dead for head 0 only
    sc.exclude_head(0, 0, np.arange(64, 96), 0)
    sc.exclude_head(0, 0, np.arange(64, 96), 1)                        # page 2: dead for both heads
    sc.leave_out(0, 0, np.arange(96, 132))                             # partial INT4 page and staging: all dead
    sc.drop()
    sc.sync()
    sc.check_tables()
    assert sc.gpu[0].info(g)[0] == 4                                   # pages 0, 1, the partial page, staging
    sc.decode(0, "partial and per-head pages kept")


def test_drop_validates_before_any_change(kvq):
    sc = Groups(kvq, [1], 4, [np.full(64, 4, np.uint8)])
    g = sc.g_ids[0][0]
    sc.gpu[0].evict(np.full(32, g), np.arange(32))
    with pytest.raises(kvq.KVError):
        sc.gpu[0].drop_dead_pages([g, 77])
    sc.sync()
    assert sc.gpu[0].info(g)[0] == 2
    sc.gpu[0].drop_dead_pages([])
    sc.gpu[0].drop_dead_pages([g])
    sc.sync()
    assert sc.gpu[0].info(g)[0] == 1


# ---- kv_decode_attn_groups ------------------------------------------------

@pytest.mark.parametrize("groups,hq,keep", [
    ([2, 2], 8, [1.0, 0.4]),                        # g = 2 (paired columns)
    ([1, 2, 1], 32, [0.25, 1.0, 0.6]),              # g = 8
    ([4], 16, [0.5]),                               # one pool: the grouped scan alone
    ([1] * 8, 8, [1.0, 0.9, 0.7, 0.5, 0.3, 0.2, 0.1, 0.0]),   # g = 1, eight pools, one keeps nothing
    ([8] * 8, 512, [1.0, 0.8, 0.6, 0.5, 0.4, 0.3, 0.2, 0.1]),  # g = 8, eight pools of 8: 64 kv heads
])
def test_grouped_decode_matches_shared_pool(kvq, groups, hq, keep):
    """Each group keeps the most recent keep[j] of every request, evicts the
    rest and drops its dead pages; group 0 also excludes a random tenth of
    the positions for its first kv head.  One grouped decode over the pools
    against S; then a decode step's tokens are appended to every pool (the
    cached plan grows) and the decode repeated."""
    rng = np.random.default_rng(len(groups) * 100 + hq)
    bits = [_mixed(520, 0.6, 3), _mixed(333, 0.5, 4), _mixed(1000, 0.7, 5)]
    sc = Groups(kvq, groups, hq, bits, stream0=10, extra=12)
    for r, n in enumerate(sc.n_tok):
        for j, kf in enumerate(keep):
            sc.leave_out(j, r, np.arange(n - int(round(kf * n))))
        sc.exclude_head(0, r, np.sort(rng.choice(n, n // 10, replace=False)), 0)
    sc.reorder()
    sc.drop()
    sc.sync()
    sc.check_tables()
    sc.decode(0, f"groups={groups}")
    for step in range(1, 4):
        for r in range(len(bits)):
            sc.append(r, _mixed(1, 0.5, 100 * step + r))
        sc.sync()
        sc.decode(step, f"groups={groups} step {step}")
    # a new page (the 33rd token of a fresh INT4 run) after the plan was cached
    for r in range(len(bits)):
        sc.append(r, np.full(40, 4, np.uint8))
    sc.sync()
    sc.check_tables(content=False)
    sc.decode(9, f"groups={groups} after 40 appends")


@pytest.mark.parametrize("groups,hq", [([2, 2], 8), ([1, 2, 1], 32)])
def test_grouped_decode_with_int3_and_fp4_pages(kvq, groups, hq):
    """Group pools holding INT2, INT3, INT4 and FP4 pages (the grouped scan's
    variant that reads them), budgets per group, a drop, then decode steps."""
    rng = np.random.default_rng(len(groups))
    widths = np.array([2, 3, 4, 0xF4], np.uint8)
    bits = [rng.choice(widths, n, p=[0.4, 0.2, 0.2, 0.2]) for n in (520, 333, 900)]
    sc = Groups(kvq, groups, hq, bits, stream0=30, extra=12)
    keep = [1.0, 0.5, 0.3][:len(groups)]
    for r, n in enumerate(sc.n_tok):
        for j, kf in enumerate(keep):
            sc.leave_out(j, r, np.arange(n - int(round(kf * n))))
    sc.reorder()
    sc.drop()
    sc.sync()
    sc.check_tables()
    sc.decode(0, f"four widths groups={groups}")
    for step in range(1, 4):
        for r in range(len(bits)):
            sc.append(r, rng.choice(widths, 1))
        sc.sync()
        sc.decode(step, f"four widths groups={groups} step {step}")


def test_grouped_decode_stats_count_only_pages_read(kvq):
    """kv_last_decode_stats after a grouped decode: a pool that dropped or
    skips pages reports fewer bytes than one that reads every page."""
    bits = [_mixed(640, 0.5, 7)]
    sc = Groups(kvq, [2, 2], 8, bits)
    sc.leave_out(1, 0, np.arange(480))
    sc.reorder()
    sc.sync()
    sc.decode(0, "stats, before drop")
    b_full = sc.gpu[0].last_decode_stats()["kv_bytes"]
    b_short = sc.gpu[1].last_decode_stats()["kv_bytes"]
    assert b_short < b_full / 2
    n0 = sc.gpu[1].info(sc.g_ids[1][0])[0]
    sc.drop()
    sc.sync()
    n1 = sc.gpu[1].info(sc.g_ids[1][0])[0]
    assert n1 < n0
    sc.decode(1, "stats, after drop")
    # the dropped pages were skipped already: only their 8-byte table entries go
    assert sc.gpu[1].last_decode_stats()["kv_bytes"] == b_short - 8 * (n0 - n1)
    assert sc.gpu[0].last_decode_stats()["kv_bytes"] == b_full


def test_grouped_decode_rejects_bad_calls(kvq):
    sc = Groups(kvq, [2, 2], 8, [np.full(64, 4, np.uint8)])
    qh, qd = _q(1, 8, 0)
    ids = np.array(sc.g_ids, np.int32)
    G = kvq.KVPool.decode_groups
    with pytest.raises(kvq.KVError):
        G([sc.gpu[0], sc.gpu[0]], qd, ids, SCALE)                      # a pool listed twice
    with pytest.raises(kvq.KVError):
        G(sc.gpu, _q(1, 6, 0)[1], ids, SCALE)                          # 6 q heads over 4 kv heads
    with pytest.raises(kvq.KVError):
        G(sc.gpu, qd, np.array([[sc.g_ids[0][0]], [5]], np.int32), SCALE)   # request not open
    with pytest.raises(ValueError):
        G(sc.gpu, qd, ids[:1], SCALE)                                  # req_ids not [n_pools][B]
    sc.gpu[1].fp_configure(64)
    k, v = _rows(3, 2, 50)
    sc.gpu[1].fp_append(sc.g_ids[1][0], _dev(k), _dev(v))
    with pytest.raises(kvq.KVError):
        G(sc.gpu, qd, ids, SCALE)                                      # full-precision tokens are not read
    sc.gpu[1].fp_drop(sc.g_ids[1][0], 0, 3)
    sc.sync()
    sc.decode(0, "after the rejected calls")


def test_config2_full_size_head_groups(kvq):
    """The 32K-token batch-8 workload (8 kv heads) as 2 head-group pools built,
    evicted and dropped exactly as `bench.py --head-groups 2` builds them
    (group 0 keeps the most recent half of every prompt, group 1 all of it),
    then 3 decode steps.  Oracle twins model each group's pool as a shared
    pool over all heads with the group's positions evicted and its dead pages
    dropped (ids and tables do not depend on the heads a pool holds): every
    table of both pools bit-exact, sampled units' codes and outputs within the
    tolerance."""
    from harness import OracleWorkload, oracle_bits
    from mixed_precision_kv_gb300.workload import GroupWorkload, pool_size
    steps = 3
    w = kvsynth.make_workload(2, steps=steps)
    G = GroupWorkload(w, 2, steps=steps)
    for r in range(len(w.requests)):
        assert np.array_equal(G.bits[r], oracle_bits(w, r))
    G.prefill()
    G.evict_and_drop()
    G.sync()
    sampled = {0: [1], 1: [6]}   # global kv heads (group 0: heads 0-3, group 1: heads 4-7)
    reqs = [0, 5]
    twins = []
    for j in range(2):
        ow = OracleWorkload(w, pool_size(w, G.bits, G.chunk, G.gw.steps), G.chunk, sel_heads=sampled[j],
                            content_reqs=reqs)
        ow.prefill()
        for r in range(len(w.requests)):
            pos = G.cut(r, j)
            assert ow.P.evict(np.full(pos.size, ow.rids[r]), pos) == oracle.OK
        ow.reorder()
        assert ow.P.drop_dead_pages(ow.rids) == oracle.OK
        twins.append(ow)
    B, g = len(w.requests), w.g

    def check(step, content):
        out = G.decode(G.q(step)).cpu().numpy()
        G.sync()
        for j, ow in enumerate(twins):
            for r in range(B):
                compare_tables(G.pools[j].export(int(G.rids[j][r]), content=False),
                               ow.P.export(ow.rids[r], content=False))
            if content:
                for r in reqs:
                    compare_content(G.pools[j].export(int(G.rids[j][r])), ow.P.export(ow.rids[r]),
                                    [h - G.lo[j] for h in sampled[j]])
            pairs = np.array([(b, h * g + x) for b in reqs for h in sampled[j] for x in range(g)], np.int32)
            ref = ow.decode(ow.q(step), pairs=pairs)
            got = np.stack([out[b, hq] for b, hq in pairs])
            assert np.isfinite(got).all()
            assert_outputs_close(got, ref, f"32K batch 8, group {j}, step {step}")

    check(0, True)
    for step in range(1, steps + 1):
        k, v, bits = G.step_inputs()
        G.append_step(k, v, bits)
        for ow in twins:
            ow.append_step()
            ow.reorder()
        check(step, step == steps)
