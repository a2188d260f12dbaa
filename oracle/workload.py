"""Oracle pools for samples of a kvsynth workload (test infrastructure: used
by the benchmark's CPU-baseline leg and its reference arm)."""
from __future__ import annotations

import numpy as np

import kvsynth
from kvsynth.recipes import tag_counts

from . import OK, OraclePool, alloc_bits


class OracleRequest:
    def __init__(self, P, rid, w):
        self.P, self.rids, self.w = P, [rid], w

    def q(self, step):
        return kvsynth.fill_bf16_host(len(self.w.requests), self.w.num_q_heads, 128, self.w.seed,
                                      kvsynth.TENSOR_Q, step)


def request_bits(w, r):
    """Bit width of every prefill position of request r (greedy allocation over its tags)."""
    spec = w.requests[r]
    b = alloc_bits(tag_counts(spec.tags[:spec.n_prefill]), w.D2, w.D4, spec.budget)
    return b[spec.tags[:spec.n_prefill]].astype(np.uint8)


def kv_rows(w, r, tok0, n, heads):
    """bf16 K and V rows [n][len(heads)][128] of request r from position tok0."""
    spec = w.requests[r]
    rm = None if spec.row_mult is None else spec.row_mult[tok0:tok0 + n]
    k = kvsynth.fill_bf16_host_heads(n, w.num_kv_heads, 128, w.seed, kvsynth.TENSOR_K, spec.stream, heads,
                                     tok0=tok0, chan_mult=w.k_chan_mult, row_mult=rm)
    v = kvsynth.fill_bf16_host_heads(n, w.num_kv_heads, 128, w.seed, kvsynth.TENSOR_V, spec.stream, heads,
                                     tok0=tok0, row_mult=rm)
    return k, v


def oracle_twin_for(w, r=0, chunk=16384, heads=None, n_tok=None):
    """Build request r of workload w in an oracle pool (the listed kv heads,
    all by default; its first n_tok prefill tokens, all by default), reorder
    it, and return (handle, (b=0, q head) pairs of the listed kv heads,
    algorithmic decode bytes of those units)."""
    spec = w.requests[r]
    bits = request_bits(w, r)
    n = spec.n_prefill if n_tok is None else min(n_tok, spec.n_prefill)
    H = w.num_kv_heads
    heads = list(range(H)) if heads is None else list(heads)
    n2 = int((bits[:n] == 2).sum()) // 32 + 2
    n4 = -(-int((bits[:n] == 4).sum()) // 32) + chunk // 32 + 4
    P = OraclePool(H, n2, n4, 1, n2 + n4, sel_heads=heads)
    rid = P.open()
    for t0 in range(0, n, chunk):
        m = min(chunk, n - t0)
        k, v = kv_rows(w, r, t0, m, heads)
        assert P.append(np.full(m, rid), bits[t0:t0 + m], k, v) == OK
    if spec.evict.size:
        ev = spec.evict[spec.evict < n]
        assert P.evict(np.full(ev.size, rid), ev) == OK
    assert P.reorder([rid]) == OK
    ex = P.export(rid, content=False)
    nbytes = 0
    for is2, f in zip(ex["is_int2"], ex["fill"]):
        nbytes += (3072 if is2 else 160 * int(f)) * len(heads) + 8
    nbytes += len(heads) * w.g * 128 * 6
    pairs = np.array([(0, h * w.g + j) for h in heads for j in range(w.g)], np.int32)
    return OracleRequest(P, rid, w), pairs, nbytes
