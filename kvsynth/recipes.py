"""Workload recipes: the five decode workloads (and shrunken variants of them).

Every array here is drawn from ``numpy.random.default_rng`` seeded with
``[seed, part, index]``, so each request's draws do not depend on how many
other requests exist.  Nothing here quantizes, allocates or attends.

Shapes follow the agentic long-context workloads the TriAxialKV and HyQuant
pages evaluate (contexts past 100K tokens, GQA models of the Qwen3 / Llama-3
families); the benchmarks those pages use are not available and these
synthetic inputs stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

N_TAGS = 4 * 2 * 7          # temporal x modal x semantic (TriAxialKV, key design 1)
HEAD_DIM = 128
PAGE = 32

_PART_TABLE, _PART_OUTLIER, _PART_REQ = 1, 2, 3


@dataclass
class RequestSpec:
    n_prefill: int                    # tokens appended before the first decode step
    tags: np.ndarray                  # uint8 [n_prefill + n_decode]: tag of each token position
    budget: Tuple[int, int]           # average-bit budget B as a fraction (num, den)
    row_mult: Optional[np.ndarray]    # float32 [n_prefill + n_decode] or None (x8 rows)
    evict: np.ndarray                 # int64 token positions evicted after prefill
    stream: int                       # generator stream id of this request


@dataclass
class Workload:
    name: str
    cfg_id: int
    seed: int
    num_q_heads: int
    num_kv_heads: int
    requests: List[RequestSpec]
    D2: np.ndarray                    # float64 [56]  D_k(2)
    D4: np.ndarray                    # float64 [56]  D_k(4)
    k_chan_mult: np.ndarray           # float32 [Hkv][128]  (x20 outlier K channels)
    steps: int                        # decode steps (one appended token per request per step)
    force_int4_decode: bool           # appended tokens go to INT4 regardless of tag
    head_dim: int = HEAD_DIM
    page_tokens: int = PAGE
    softmax_scale: float = float(np.float32(1.0 / np.sqrt(HEAD_DIM)))
    notes: dict = field(default_factory=dict)

    @property
    def g(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def tag_runs(rng: np.random.Generator, n: int) -> np.ndarray:
    """Tags in contiguous runs of 16..256 tokens, each run's tag uniform over the 56 tags."""
    out = np.empty(n, dtype=np.uint8)
    pos = 0
    while pos < n:
        ln = int(rng.integers(16, 257))
        out[pos:pos + ln] = int(rng.integers(0, N_TAGS))
        pos += ln
    return out


def _rng(seed, part, idx=0):
    return np.random.default_rng([seed, part, idx])


def _tables(seed):
    r = _rng(seed, _PART_TABLE)
    d4 = r.uniform(0.01, 1.0, N_TAGS)
    d2 = d4 * (1.0 + r.uniform(0.5, 20.0, N_TAGS))
    return d2, d4


def _outliers(seed, hkv):
    r = _rng(seed, _PART_OUTLIER)
    m = np.ones((hkv, HEAD_DIM), dtype=np.float32)
    for h in range(hkv):
        m[h, r.choice(HEAD_DIM, 4, replace=False)] = 20.0
    return m


_DEFAULTS = {
    1: dict(name="tiny-2k-g4", hq=8, hkv=2, n_req=1, steps=0),
    2: dict(name="qwen3-8b-32k-b8", hq=32, hkv=8, n_req=8, steps=0),
    3: dict(name="llama3-70b-100k-b16", hq=64, hkv=8, n_req=16, steps=0),
    4: dict(name="ragged-64req-1k-128k-evict5", hq=32, hkv=8, n_req=64, steps=0),
    5: dict(name="serving-256req-4k-64k-64steps", hq=32, hkv=8, n_req=256, steps=64),
}


def make_workload(cfg_id: int, n_req: Optional[int] = None, ctx: Optional[int] = None,
                  ctx_range: Optional[Tuple[int, int]] = None, steps: Optional[int] = None,
                  seed: Optional[int] = None) -> Workload:
    """Workload `cfg_id` (1..5) at full size, or shrunk via n_req / ctx / ctx_range / steps."""
    d = _DEFAULTS[cfg_id]
    seed = 1000 + cfg_id if seed is None else seed
    n_req = d["n_req"] if n_req is None else n_req
    steps = d["steps"] if steps is None else steps
    hkv = d["hkv"]
    D2, D4 = _tables(seed)
    reqs = []
    for r in range(n_req):
        rr = _rng(seed, _PART_REQ, r)
        if cfg_id == 1:
            n = 2048 if ctx is None else ctx
            budget = (3, 1)
        elif cfg_id == 2:
            n = 32768 if ctx is None else ctx
            budget = (3, 1)
        elif cfg_id == 3:
            n = 100000 if ctx is None else ctx
            budget = (5, 2)
        elif cfg_id == 4:
            lo, hi = (1024, 131072) if ctx_range is None else ctx_range
            n = int(round(np.exp(rr.uniform(np.log(lo), np.log(hi))))) if ctx is None else ctx
            f_milli = int(round(rr.uniform(0.2, 0.9) * 1000))
            budget = (4000 - 2 * f_milli, 1000)          # B_r = 4 - 2 f_r
        else:
            lo, hi = (4096, 65536) if ctx_range is None else ctx_range
            n = int(rr.integers(lo, hi + 1)) if ctx is None else ctx
            budget = (3, 1)
        total = n + steps
        tags = tag_runs(rr, total)
        row_mult = None
        if cfg_id == 3:
            row_mult = np.ones(total, dtype=np.float32)
            row_mult[rr.choice(total, max(1, total // 100), replace=False)] = 8.0
        evict = np.zeros(0, dtype=np.int64)
        if cfg_id == 4:
            evict = np.sort(rr.choice(n, int(round(0.05 * n)), replace=False)).astype(np.int64)
        reqs.append(RequestSpec(n_prefill=n, tags=tags, budget=budget, row_mult=row_mult,
                                evict=evict, stream=r))
    return Workload(name=d["name"], cfg_id=cfg_id, seed=seed, num_q_heads=d["hq"], num_kv_heads=hkv,
                    requests=reqs, D2=D2, D4=D4, k_chan_mult=_outliers(seed, hkv), steps=steps,
                    force_int4_decode=(cfg_id == 2))


def tag_counts(tags: np.ndarray) -> np.ndarray:
    return np.bincount(tags, minlength=N_TAGS).astype(np.int64)


FP4_WIDTH = 0xF4   # width value of FP4 (E2M1) tokens


def width_mix(w: Workload, r: int, bits: np.ndarray, int3_share: float, fp4_share: float = 0.0) -> np.ndarray:
    """Input recipe for workloads with more widths than the two-way
    allocation gives: a seeded fraction `int3_share` of request r's INT4
    tokens made INT3 and a further `fp4_share` made FP4 (one uniform draw per
    position, seeded by the workload seed and the request)."""
    if int3_share <= 0.0 and fp4_share <= 0.0:
        return bits
    u = np.random.default_rng([w.seed, 33, r]).random(bits.size)
    out = bits.copy()
    out[(bits == 4) & (u < int3_share)] = 3
    out[(bits == 4) & (u >= int3_share) & (u < int3_share + fp4_share)] = FP4_WIDTH
    return out


_PART_TABLE3 = 4


def d3_table(w: Workload) -> np.ndarray:
    """D_k(3) for the three-width allocation: between D_k(4) and D_k(2), the
    2 -> 3 step saving 55..80 % of the 2 -> 4 saving (a convex distortion
    curve), from its own seeded stream (the two-width tables are unchanged)."""
    r = _rng(w.seed, _PART_TABLE3)
    return w.D4 + (w.D2 - w.D4) * r.uniform(0.2, 0.45, w.D2.size)
