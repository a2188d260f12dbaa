"""Oracle pool for one request of a kvsynth workload (test infrastructure:
used by the benchmark's CPU-baseline leg and its reference arm)."""
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


def oracle_twin_for(w, r=0, chunk=16384):
    """Build request r of workload w in an oracle pool (all kv heads), reorder
    it, and return (handle, (b=0, q head) pairs, algorithmic decode bytes)."""
    spec = w.requests[r]
    b = alloc_bits(tag_counts(spec.tags[:spec.n_prefill]), w.D2, w.D4, spec.budget)
    bits = b[spec.tags[:spec.n_prefill]].astype(np.uint8)
    n = spec.n_prefill
    H = w.num_kv_heads
    n2 = int((bits == 2).sum()) // 32 + 2
    n4 = -(-int((bits == 4).sum()) // 32) + chunk // 32 + 4
    P = OraclePool(H, n2, n4, 1, n2 + n4)
    rid = P.open()
    for t0 in range(0, n, chunk):
        m = min(chunk, n - t0)
        rm = None if spec.row_mult is None else spec.row_mult[t0:t0 + m]
        k = kvsynth.fill_bf16_host(m, H, 128, w.seed, kvsynth.TENSOR_K, spec.stream, t0, chan_mult=w.k_chan_mult,
                                   row_mult=rm)
        v = kvsynth.fill_bf16_host(m, H, 128, w.seed, kvsynth.TENSOR_V, spec.stream, t0, row_mult=rm)
        assert P.append(np.full(m, rid), bits[t0:t0 + m], k, v) == OK
    if spec.evict.size:
        assert P.evict(np.full(spec.evict.size, rid), spec.evict) == OK
    assert P.reorder([rid]) == OK
    ex = P.export(rid, content=False)
    nbytes = 0
    for is2, f in zip(ex["is_int2"], ex["fill"]):
        nbytes += (3072 if is2 else 160 * int(f)) * H + 8
    nbytes += w.num_q_heads * 128 * 6
    pairs = np.array([(0, h) for h in range(w.num_q_heads)], np.int32)
    return OracleRequest(P, rid, w), pairs, nbytes
