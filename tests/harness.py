"""Test harness: build the oracle's pool for a kvsynth workload with the same
append call boundaries as the GPU driver, and compare the two sides."""
from __future__ import annotations

import numpy as np

import kvsynth
import oracle
from kvsynth.recipes import d3_table, tag_counts, width_mix

MAX_ABS_TOL = 1e-3     # attention output, fp32 vs fp64 oracle on the same dequantized values
REL_L2_TOL = 1e-4


def oracle_bits(w, r, three_widths=False):
    spec = w.requests[r]
    if three_widths:
        b = oracle.alloc_bits3(tag_counts(spec.tags[:spec.n_prefill]), w.D2, d3_table(w), w.D4, spec.budget)
    else:
        b = oracle.alloc_bits(tag_counts(spec.tags[:spec.n_prefill]), w.D2, w.D4, spec.budget)
    bits = b[spec.tags].astype(np.uint8)
    if w.force_int4_decode:
        bits[spec.n_prefill:] = 4
    return bits


class OracleWorkload:
    """Oracle twin of mixed_precision_kv_gb300.workload.GPUWorkload."""

    def __init__(self, w, sizes, chunk, sel_heads=None, content_reqs=None, n_int3_pages=0, n_fp4_pages=0,
                 int3_share=0.0, fp4_share=0.0, three_widths=False):
        n2, n4, max_tab = sizes
        self.w = w
        self.chunk = chunk
        self.sel = list(range(w.num_kv_heads)) if sel_heads is None else list(sel_heads)
        self.content = set(range(len(w.requests))) if content_reqs is None else set(content_reqs)
        self.P = oracle.OraclePool(w.num_kv_heads, n2, n4, len(w.requests), max_tab, sel_heads=self.sel,
                                   n_int3_pages=n_int3_pages, n_fp4_pages=n_fp4_pages)
        self.rids = [self.P.open() for _ in w.requests]
        self.bits = [width_mix(w, r, oracle_bits(w, r, three_widths), int3_share, fp4_share)
                     for r in range(len(w.requests))]
        self.pos = [0] * len(w.requests)

    def kv_rows(self, r, tok0, n):
        spec = self.w.requests[r]
        rm = None if spec.row_mult is None else spec.row_mult[tok0:tok0 + n]
        H = self.w.num_kv_heads
        k = kvsynth.fill_bf16_host_heads(n, H, 128, self.w.seed, kvsynth.TENSOR_K, spec.stream, self.sel, tok0=tok0,
                                         chan_mult=self.w.k_chan_mult, row_mult=rm)
        v = kvsynth.fill_bf16_host_heads(n, H, 128, self.w.seed, kvsynth.TENSOR_V, spec.stream, self.sel, tok0=tok0,
                                         row_mult=rm)
        return k, v

    def prefill(self):
        for r, spec in enumerate(self.w.requests):
            for t0 in range(0, spec.n_prefill, self.chunk):
                n = min(self.chunk, spec.n_prefill - t0)
                k = v = None
                if r in self.content:
                    k, v = self.kv_rows(r, t0, n)
                assert self.P.append(np.full(n, self.rids[r]), self.bits[r][t0:t0 + n], k, v) == oracle.OK
            self.pos[r] = spec.n_prefill

    def evict(self):
        for r, spec in enumerate(self.w.requests):
            if spec.evict.size:
                assert self.P.evict(np.full(spec.evict.size, self.rids[r]), spec.evict) == oracle.OK

    def reorder(self):
        assert self.P.reorder(self.rids) == oracle.OK

    def append_step(self):
        ks, vs = [], []
        for r in range(len(self.rids)):
            k, v = self.kv_rows(r, self.pos[r], 1)
            ks.append(k)
            vs.append(v)
        bits = np.array([self.bits[r][self.pos[r]] for r in range(len(self.rids))], np.uint8)
        assert self.P.append(np.array(self.rids), bits, np.concatenate(ks), np.concatenate(vs)) == oracle.OK
        for r in range(len(self.rids)):
            self.pos[r] += 1

    def q(self, step):
        return kvsynth.fill_bf16_host(len(self.rids), self.w.num_q_heads, 128, self.w.seed, kvsynth.TENSOR_Q, step)

    def decode(self, q_bits, pairs=None, n_threads=0):
        return self.P.decode(q_bits, self.rids, self.w.softmax_scale, pairs=pairs, n_threads=n_threads)


def compare_tables(gpu_ex, orc_ex):
    for key in ("ids", "is_int2", "fill", "live"):
        assert np.array_equal(gpu_ex[key], orc_ex[key]), key


def compare_content(gpu_ex, orc_ex, sel):
    """Codes and binary16 scale/zero bit-exact on every written slot of the selected heads."""
    compare_tables(gpu_ex, orc_ex)
    for i in range(orc_ex["ids"].size):
        f = int(orc_ex["fill"][i])
        for j, h in enumerate(sel):
            assert np.array_equal(gpu_ex["kc"][i, h, :f], orc_ex["kc"][i, j, :f]), (i, h, "k codes")
            assert np.array_equal(gpu_ex["vc"][i, h, :f], orc_ex["vc"][i, j, :f]), (i, h, "v codes")
            gk, ok = gpu_ex["km"][i, h], orc_ex["km"][i, j]
            gv, ov = gpu_ex["vm"][i, h], orc_ex["vm"][i, j]
            if orc_ex["is_int2"][i]:
                assert np.array_equal(gk, ok), (i, h, "k meta")
            else:
                assert np.array_equal(gk[:8 * f], ok[:8 * f]), (i, h, "k meta")
            assert np.array_equal(gv[:8 * f], ov[:8 * f]), (i, h, "v meta")


def output_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.abs(got - ref).max()) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel


def assert_outputs_close(got, ref, what=""):
    max_abs, rel = output_errors(got, ref)
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel
