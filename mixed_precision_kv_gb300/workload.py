"""Drive a KVPool through a synthetic decode workload (kvsynth recipe).

Everything here goes through the public binding: bit allocation with
``alloc_bits``, prefill and per-step appends with ``KVPool.append``, eviction,
reorder and decode.  Inputs are generated on the device by kvsynth's
counter-based generator, so a CPU checker can regenerate any row it samples.
"""
from __future__ import annotations

import numpy as np

import kvsynth
from kvsynth.recipes import FP4_WIDTH, Workload, d3_table, tag_counts, width_mix

from . import KVPool, alloc_bits, alloc_bits3


def request_bits(w: Workload, r: int, allocator=alloc_bits, three_widths: bool = False) -> np.ndarray:
    """Bit width of every token position of request r (prefill and decode
    steps); three_widths: the INT2/INT3/INT4 allocation over the same budget."""
    spec = w.requests[r]
    if three_widths:
        b = alloc_bits3(tag_counts(spec.tags[:spec.n_prefill]), w.D2, d3_table(w), w.D4, spec.budget)
    else:
        b = allocator(tag_counts(spec.tags[:spec.n_prefill]), w.D2, w.D4, spec.budget)
    bits = b[spec.tags].astype(np.uint8)
    if w.force_int4_decode:
        bits[spec.n_prefill:] = 4
    return bits


FP4 = FP4_WIDTH   # width value of FP4 (E2M1) tokens


def int3_pages(w: Workload, bits_list, steps: int, width: int = 3) -> int:
    """Pages the workload's tokens of one tail width (INT3 or FP4) take
    (prefill and steps)."""
    n3 = 0
    for spec, bits in zip(w.requests, bits_list):
        b3 = int((bits[:spec.n_prefill + steps] == width).sum())
        n3 += -(-b3 // 32) + 1 if b3 else 0
    return n3


def pool_size(w: Workload, bits_list, chunk: int, steps: int, extra: int = 0):
    """INT2 / INT4 page counts and table capacity for a workload appended in
    `chunk`-token calls and then `steps` one-token-per-request calls, with room
    for `extra` more tokens per request of either width (INT3 pages:
    int3_pages)."""
    n2 = n4 = max_tab = 0
    xp = -(-extra // 32) + 1 if extra else 0
    for spec, bits in zip(w.requests, bits_list):
        total = spec.n_prefill + steps
        b2 = int((bits[:total] == 2).sum())
        b3 = int((bits[:total] == 3).sum()) + int((bits[:total] == FP4).sum())
        b4 = total - b2 - b3
        n2 += b2 // 32 + 1 + xp
        n4 += -(-b4 // 32) + 2 + xp
        max_tab = max(max_tab, b2 // 32 + -(-b4 // 32) + -(-b3 // 32) + 3 + 2 * xp)
    # staging pages repacked during one call are freed only when it returns
    n4 += chunk // 32 + len(w.requests) + 8
    return n2, n4, max_tab


class GPUWorkload:
    def __init__(self, w: Workload, device: int = 0, chunk: int = 16384, steps: int | None = None,
                 extra_tokens: int = 0, make_pool: bool = True, int3_share: float = 0.0, fp4_share: float = 0.0,
                 three_widths: bool = False):
        import torch
        self.w = w
        self.device = device
        self.chunk = chunk
        self.steps = w.steps if steps is None else steps
        self.bits = [width_mix(w, r, request_bits(w, r, three_widths=three_widths), int3_share, fp4_share)
                     for r in range(len(w.requests))]
        self.sizes = pool_size(w, self.bits, chunk, self.steps, extra_tokens)
        n2, n4, max_tab = self.sizes
        n3 = int3_pages(w, self.bits, self.steps)
        nf = int3_pages(w, self.bits, self.steps, FP4)
        # make_pool=False: the caller builds its own pools (e.g. one per head
        # group) and uses this object for the bit allocation and the rows
        self.pool = (KVPool(w.num_kv_heads, n2, n4, len(w.requests), max_tab, device=device, n_int3_pages=n3,
                            n_fp4_pages=nf) if make_pool else None)
        self.rids = [self.pool.open() for _ in w.requests] if make_pool else []
        self.dev = torch.device("cuda", device)
        self.chan = torch.from_numpy(w.k_chan_mult).to(self.dev)
        self.row = [None if s.row_mult is None else torch.from_numpy(s.row_mult).to(self.dev) for s in w.requests]
        self.pos = [0] * len(w.requests)

    def _gen(self, n, tensor, stream, tok0, chan, row):
        import torch
        H = self.w.num_kv_heads
        out = torch.empty((n, H, 128), dtype=torch.bfloat16, device=self.dev)
        kvsynth.fill_bf16_dev(out.data_ptr(), n, H, 128, self.w.seed, tensor, stream, tok0,
                              chan.data_ptr() if chan is not None else 0,
                              row[tok0:tok0 + n].data_ptr() if row is not None else 0,
                              torch.cuda.current_stream(self.dev).cuda_stream)
        return out

    def kv_rows(self, r, tok0, n):
        spec = self.w.requests[r]
        k = self._gen(n, kvsynth.TENSOR_K, spec.stream, tok0, self.chan, self.row[r])
        v = self._gen(n, kvsynth.TENSOR_V, spec.stream, tok0, None, self.row[r])
        return k, v

    def prefill(self):
        for r, spec in enumerate(self.w.requests):
            for t0 in range(0, spec.n_prefill, self.chunk):
                n = min(self.chunk, spec.n_prefill - t0)
                k, v = self.kv_rows(r, t0, n)
                self.pool.append(k, v, np.full(n, self.rids[r], np.int32), self.bits[r][t0:t0 + n])
            self.pos[r] = spec.n_prefill

    def evict(self):
        for r, spec in enumerate(self.w.requests):
            if spec.evict.size:
                self.pool.evict(np.full(spec.evict.size, self.rids[r], np.int32), spec.evict)

    def reorder(self):
        self.pool.reorder(self.rids)

    def q(self, step: int):
        import torch
        Hq = self.w.num_q_heads
        out = torch.empty((len(self.rids), Hq, 128), dtype=torch.bfloat16, device=self.dev)
        kvsynth.fill_bf16_dev(out.data_ptr(), len(self.rids), Hq, 128, self.w.seed, kvsynth.TENSOR_Q, step, 0,
                              0, 0, torch.cuda.current_stream(self.dev).cuda_stream)
        return out

    def step_inputs(self):
        """K/V [B][Hkv][128] of the next token of every request, plus its req ids and bits."""
        import torch
        ks, vs = [], []
        for r in range(len(self.rids)):
            k, v = self.kv_rows(r, self.pos[r], 1)
            ks.append(k)
            vs.append(v)
        bits = np.array([self.bits[r][self.pos[r]] for r in range(len(self.rids))], np.uint8)
        return torch.cat(ks), torch.cat(vs), np.array(self.rids, np.int32), bits

    def append_step(self, k, v, req_ids, bits):
        self.pool.append(k, v, req_ids, bits)
        for r in range(len(self.rids)):
            self.pos[r] += 1

    def freeze_segments(self, rho: float = 0.05, window: int = 128, staging: int = 128):
        """Full-precision segments on the prefilled pool (HyQuant, Algorithm 4
        FREEZE): per request and kv head the top-rho positions of a seeded
        synthetic column score over the non-window prefix leave that head's
        quantized set (per-head exclusion) for its full-precision list; the
        last `window` prefill positions leave every head's quantized set
        (eviction) and follow in the lists.  The lists hold room for the
        staging buffer.  Returns the window tokens' rows [window][B][Hkv][128]
        (K, V) and the number of vertical-line tokens per request."""
        import torch
        H, B = self.w.num_kv_heads, len(self.rids)
        n_vl = [int(rho * (spec.n_prefill - window)) for spec in self.w.requests]
        self.pool.fp_configure(max(n_vl) + window + staging)
        wk = torch.empty((window, B, H, 128), dtype=torch.bfloat16, device=self.dev)
        wv = torch.empty_like(wk)
        for r, spec in enumerate(self.w.requests):
            n, pre, nv = spec.n_prefill, spec.n_prefill - window, n_vl[r]
            rid = self.rids[r]
            k_all, v_all = self.kv_rows(r, 0, n)
            score = np.random.default_rng([self.w.seed, 77, r]).random((H, pre))
            pos = [np.sort(np.argpartition(score[h], pre - nv)[pre - nv:]) for h in range(H)]
            idx = [torch.from_numpy(p_).to(self.dev) for p_ in pos]
            kf = torch.stack([k_all[idx[h], h] for h in range(H)], dim=1).contiguous()
            vf = torch.stack([v_all[idx[h], h] for h in range(H)], dim=1).contiguous()
            self.pool.evict_head(np.full(nv * H, rid), np.concatenate(pos), np.repeat(np.arange(H), nv))
            self.pool.evict(np.full(window, rid), np.arange(pre, n))
            self.pool.fp_append(rid, kf, vf)
            self.pool.fp_append(rid, k_all[pre:n].contiguous(), v_all[pre:n].contiguous())
            wk[:, r] = k_all[pre:n]
            wv[:, r] = v_all[pre:n]
        return wk, wv, n_vl

    def decode(self, q, out=None):
        return self.pool.decode(q, self.rids, self.w.softmax_scale, out=out)

    def kv_bytes(self) -> int:
        return self.pool.last_decode_stats()["kv_bytes"]


class GroupWorkload:
    """The workload's kv heads cut into `n_groups` equal head groups, one pool
    each (Tangram: head groups keep different amounts of context), fed the
    group's rows of every token in the same calls.  Group j keeps the most
    recent keep[j] of every prompt (default (j + 1) / n_groups): its pool
    evicts the older positions (and the workload's own evictions) and drops
    the pages no kv head of the group reads any more."""

    def __init__(self, w: Workload, n_groups: int, device: int = 0, chunk: int = 16384, steps: int | None = None,
                 keep=None):
        import torch
        H = w.num_kv_heads
        if n_groups < 1 or n_groups > 8 or H % n_groups:
            raise ValueError("n_groups must divide the kv heads, at most 8 groups")
        self.w, self.N, self.hg = w, n_groups, H // n_groups
        self.lo = [j * self.hg for j in range(n_groups + 1)]
        self.keep = [(j + 1) / n_groups for j in range(n_groups)] if keep is None else list(keep)
        self.gw = GPUWorkload(w, device=device, chunk=chunk, steps=steps, make_pool=False)
        self.bits, self.chunk, self.dev = self.gw.bits, chunk, self.gw.dev
        n2, n4, max_tab = self.gw.sizes
        self.pools = [KVPool(self.hg, n2, n4, len(w.requests), max_tab, device=device) for _ in range(n_groups)]
        self.rids = [np.array([p.open() for _ in w.requests], np.int32) for p in self.pools]
        self.pos = [0] * len(w.requests)
        self.torch = torch

    def rows(self, k, j):
        return k[:, self.lo[j]:self.lo[j + 1]].contiguous()

    def prefill(self):
        for r, spec in enumerate(self.w.requests):
            for t0 in range(0, spec.n_prefill, self.chunk):
                n = min(self.chunk, spec.n_prefill - t0)
                k, v = self.gw.kv_rows(r, t0, n)
                for j, p in enumerate(self.pools):
                    p.append(self.rows(k, j), self.rows(v, j), np.full(n, self.rids[j][r], np.int32),
                             self.bits[r][t0:t0 + n])
            self.pos[r] = spec.n_prefill

    def cut(self, r, j):
        """Positions group j leaves out of request r's prompt."""
        spec = self.w.requests[r]
        n = spec.n_prefill
        return np.union1d(spec.evict, np.arange(n - int(round(n * self.keep[j])), dtype=np.int64))

    def evict_and_drop(self):
        for r in range(len(self.w.requests)):
            for j, p in enumerate(self.pools):
                pos = self.cut(r, j)
                if pos.size:
                    p.evict(np.full(pos.size, self.rids[j][r], np.int32), pos)
        for j, p in enumerate(self.pools):
            p.reorder(self.rids[j])
            p.drop_dead_pages(self.rids[j])

    def blocks(self):
        """(page, kv head) blocks the group pools hold."""
        return sum(p.info(int(x))[0] * self.hg for p, rs in zip(self.pools, self.rids) for x in rs)

    def append_step(self, k, v, bits):
        """One token per request: k, v [B][Hkv][128] on the device."""
        for j, p in enumerate(self.pools):
            p.append(self.rows(k, j), self.rows(v, j), self.rids[j], bits)
            p.reorder(self.rids[j])
        for r in range(len(self.pos)):
            self.pos[r] += 1

    def step_inputs(self):
        ks, vs = [], []
        for r in range(len(self.w.requests)):
            k, v = self.gw.kv_rows(r, self.pos[r], 1)
            ks.append(k)
            vs.append(v)
        bits = np.array([self.bits[r][self.pos[r]] for r in range(len(self.w.requests))], np.uint8)
        return self.torch.cat(ks), self.torch.cat(vs), bits

    def q(self, step: int):
        torch = self.torch
        B, Hq = len(self.w.requests), self.w.num_q_heads
        out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device=self.dev)
        kvsynth.fill_bf16_dev(out.data_ptr(), B, Hq, 128, self.w.seed, kvsynth.TENSOR_Q, step, 0, 0, 0,
                              torch.cuda.current_stream(self.dev).cuda_stream)
        return out

    def decode(self, q, out=None):
        return KVPool.decode_groups(self.pools, q, np.stack(self.rids), self.w.softmax_scale, out=out)

    def sync(self):
        for p in self.pools:
            p.sync()
