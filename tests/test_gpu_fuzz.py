"""Seeded random sequences of pool calls, in lock step on the GPU pool and the
oracle: opens and closes, appends of every shape (one request's chunk, runs of
several requests, tokens of several requests interleaved, short calls),
evictions by position for all heads and for one head, dead-page drops and
reorders, with pools small enough that calls run out of pages or table
entries.  After every call: the same status on both sides and every open
request's table bit-exact; every few calls: codes and scale/zero of one
request, and the decode of all open requests within max-abs 1e-3 /
relative-L2 1e-4 of the fp64 oracle."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close, compare_content, compare_tables

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 6161
SCALE = float(np.float32(1 / np.sqrt(128)))
HKV, HQ = 2, 8
MAX_REQ = 6


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


FP_CAP = 256   # full-precision list capacity (segments variant)


class Lockstep:
    def __init__(self, kvq, widths, n2, n4, n3, nf, max_tab, segments=False):
        self.kvq = kvq
        self.gpu = kvq.KVPool(HKV, n2, n4, MAX_REQ, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        self.orc = oracle.OraclePool(HKV, n2, n4, MAX_REQ, max_tab, n_int3_pages=n3, n_fp4_pages=nf)
        if segments:
            self.gpu.fp_configure(FP_CAP)
        self.widths = np.array(widths, np.uint8)
        self.open_ = {}     # gpu id -> [oracle id, tokens appended, data stream]
        self.fp = {}        # gpu id -> [list tokens now, list tokens ever appended]
        self.streams = 0

    def open(self):
        g, o = self.gpu.open(), self.orc.open()
        self.open_[g] = [o, 0, self.streams]
        self.fp[g] = [0, 0]
        self.streams += 1

    def close(self, g):
        self.gpu.close_request(g)
        self.orc.close_request(self.open_.pop(g)[0])
        del self.fp[g]

    def fp_append(self, g, n):
        o, _, st = self.open_[g]
        n = min(n, FP_CAP - self.fp[g][0])
        if n <= 0:
            return
        t0 = 1_000_000 + self.fp[g][1]   # list tokens draw from their own positions of the stream
        k = kvsynth.fill_bf16_host(n, HKV, 128, SEED, kvsynth.TENSOR_K, st, t0)
        v = kvsynth.fill_bf16_host(n, HKV, 128, SEED, kvsynth.TENSOR_V, st, t0)
        self.gpu.fp_append(g, _dev(k), _dev(v))
        assert self.orc.fp_append(o, k, v) == oracle.OK
        self.fp[g][0] += n
        self.fp[g][1] += n

    def fp_drop(self, g, rng):
        cnt = self.fp[g][0]
        if cnt == 0:
            return
        first = int(rng.integers(0, cnt))
        n = int(rng.integers(1, cnt - first + 1))
        self.gpu.fp_drop(g, first, n)
        assert self.orc.fp_drop(self.open_[g][0], first, n) == oracle.OK
        self.fp[g][0] -= n

    def append(self, runs, rng, interleave=False):
        """runs: [(gpu id, n tokens)]; interleave: tokens of the runs shuffled
        into one sequence (each request's tokens keep their order)."""
        order = np.concatenate([np.full(n, i) for i, (_, n) in enumerate(runs)])
        if interleave:
            rng.shuffle(order)
        n = order.size
        k = np.empty((n, HKV, 128), np.uint16)
        v = np.empty_like(k)
        bits = self.widths[rng.integers(0, self.widths.size, n)]
        greq, oreq = np.empty(n, np.int32), np.empty(n, np.int32)
        for i, (g, m) in enumerate(runs):
            o, pos, st = self.open_[g]
            sel = np.nonzero(order == i)[0]
            k[sel] = kvsynth.fill_bf16_host(m, HKV, 128, SEED, kvsynth.TENSOR_K, st, pos)
            v[sel] = kvsynth.fill_bf16_host(m, HKV, 128, SEED, kvsynth.TENSOR_V, st, pos)
            greq[sel], oreq[sel] = g, o
        try:
            self.gpu.append(_dev(k), _dev(v), greq, bits)
            gs = 0
        except self.kvq.KVError as e:
            gs = e.status
        os_ = self.orc.append(oreq, bits, k, v)
        assert gs == os_, (gs, os_)
        if gs == 0:
            for g, m in runs:
                self.open_[g][1] += m
        return gs

    def evict(self, g, pos, heads=None):
        o = self.open_[g][0]
        if heads is None:
            self.gpu.evict(np.full(pos.size, g), pos)
            assert self.orc.evict(np.full(pos.size, o), pos) == oracle.OK
        else:
            self.gpu.evict_head(np.full(pos.size, g), pos, heads)
            assert self.orc.evict_head(np.full(pos.size, o), pos, heads) == oracle.OK

    def drop(self, gs):
        self.gpu.drop_dead_pages(gs)
        assert self.orc.drop_dead_pages([self.open_[g][0] for g in gs]) == oracle.OK

    def reorder(self):
        gs = list(self.open_)
        self.gpu.reorder(gs)
        assert self.orc.reorder([self.open_[g][0] for g in gs]) == oracle.OK

    def check_tables(self, what):
        self.gpu.sync()
        for g, (o, n, _) in self.open_.items():
            assert self.gpu.info(g)[1] == n and self.orc.info(o)[1] == n, what
            assert self.gpu.fp_count(g) == self.fp[g][0], what
            compare_tables(self.gpu.export(g, content=False), self.orc.export(o, content=False))

    def check_decode(self, rng, what):
        if not self.open_:
            return
        self.reorder()
        gs = list(self.open_)
        g = gs[int(rng.integers(0, len(gs)))]
        compare_content(self.gpu.export(g), self.orc.export(self.open_[g][0]), list(range(HKV)))
        B = len(gs)
        q = kvsynth.fill_bf16_host(B, HQ, 128, SEED, kvsynth.TENSOR_Q, int(rng.integers(0, 1 << 20)))
        out = self.gpu.decode(_dev(q), gs, SCALE).cpu().numpy()
        assert np.isfinite(out).all(), what
        ref = self.orc.decode(q, [self.open_[x][0] for x in gs], SCALE).reshape(B, HQ, 128)
        assert_outputs_close(out, ref, what)


@pytest.mark.parametrize("seed,widths,segments", [(1, [2, 4], False), (2, [2, 4], False), (3, [2, 4], False),
                                                  (4, [2, 4], False), (5, [2, 3, 4, 0xF4], False),
                                                  (6, [2, 3, 4, 0xF4], False), (7, [2, 4], True),
                                                  (8, [2, 3, 4, 0xF4], True)])
def test_random_call_sequences(kvq, seed, widths, segments):
    """segments: full-precision list appends and drops join the calls (the
    decode then scans the lists after the quantized pages)."""
    rng = np.random.default_rng([91, seed])
    L = Lockstep(kvq, widths, n2=40, n4=70, n3=24, nf=24, max_tab=30, segments=segments)
    outcomes = {"ok": 0, "oom": 0}
    ops = ["open", "close", "bulk", "runs", "interleaved", "short", "evict", "evict_head", "drop", "reorder",
           "fp_append", "fp_drop"]
    p = np.array([0.08, 0.05, 0.2, 0.17, 0.12, 0.1, 0.1, 0.08, 0.05, 0.05] + ([0.1, 0.05] if segments else [0, 0]))
    for step in range(200):
        ids = list(L.open_)
        op = rng.choice(ops, p=p / p.sum())
        if op == "open" or not ids:
            if len(L.open_) < MAX_REQ:
                L.open()
        elif op == "close":
            L.close(ids[int(rng.integers(0, len(ids)))])
        elif op in ("bulk", "short"):
            g = ids[int(rng.integers(0, len(ids)))]
            n = int(rng.integers(32, 260)) if op == "bulk" else int(rng.integers(1, 32))
            outcomes["ok" if L.append([(g, n)], rng) == 0 else "oom"] += 1
        elif op in ("runs", "interleaved"):
            m = min(len(ids), int(rng.integers(2, 4)))
            pick = rng.choice(ids, m, replace=False)
            runs = [(int(g), int(rng.integers(32, 110) if op == "runs" else rng.integers(1, 40))) for g in pick]
            outcomes["ok" if L.append(runs, rng, interleave=(op == "interleaved")) == 0 else "oom"] += 1
        elif op in ("evict", "evict_head"):
            g = ids[int(rng.integers(0, len(ids)))]
            n = L.open_[g][1]
            if n:
                pos = rng.choice(n, min(n, int(rng.integers(1, 40))), replace=False).astype(np.int64)
                heads = rng.integers(0, HKV, pos.size).astype(np.int32) if op == "evict_head" else None
                L.evict(g, pos, heads)
        elif op == "drop":
            L.drop([int(x) for x in rng.choice(ids, int(rng.integers(1, len(ids) + 1)), replace=False)])
        elif op == "fp_append":
            L.fp_append(ids[int(rng.integers(0, len(ids)))], int(rng.integers(1, 60)))
        elif op == "fp_drop":
            L.fp_drop(ids[int(rng.integers(0, len(ids)))], rng)
        else:
            L.reorder()
        L.check_tables(f"seed {seed} step {step} ({op})")
        if step % 9 == 8:
            L.check_decode(rng, f"seed {seed} step {step}")
    L.check_decode(rng, f"seed {seed} end")
    assert outcomes["ok"] >= 40 and outcomes["oom"] >= 10, outcomes   # (measured: 49..91 and 15..78)
