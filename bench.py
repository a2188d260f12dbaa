"""Benchmark: one decode step of the mixed INT2/INT4 paged-KV path.

A step = append one new token per request (quantize-on-append) + INT2-first
reorder + split-KV fused-dequant decode attention with log-sum-exp merge.  The
default workload is the Llama-3-70B-shaped single layer at long agentic
context (batch 16, 64 query / 8 KV heads, head_dim 128, 100K tokens per
request, INT2:INT4 from the greedy allocator at B = 2.5, 1 % of token rows
x8); `--config N` selects another of the five workloads.  The metric is
algorithmic KV bytes per step (codes + binary16 scale/zero of every page block
read, table entries, q, out) divided by the step time.

Launch: `python bench.py [--gpus 1] [--steps K] [--warmup W]`; for N > 1 under
torchrun each rank runs its own replica of the workload (requests are
independent; there is no data-path collective) and rank 0 reports the total.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mixed INT2/INT4 paged decode: KV-bytes GB/s (% of HBM peak), µs/layer-step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock, utilization and throttle reasons, taken
    from before the warm-up to the end of the timed region; the summary keeps
    the samples taken while the GPU was busy."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index, period_ms=20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.period), "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)
            self.proc = None

    def __enter__(self):
        return self.start()

    def __exit__(self, *a):
        self.stop()

    def summary(self):
        sm, mx, reasons, busy = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[9]), f[5:9]))
            except ValueError:
                continue
        loaded = [r for r in rows if r[2] > 0]
        for clk, cmax, _, rs in (loaded or rows):
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, rs):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "window": "from before the warm-up to the end of the timed region, every %d ms" % self.period}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_time(t_ms, dist=None, device="cpu"):
    """Job time = the slowest rank's time (all ranks run the same number of steps)."""
    if dist is None:
        return t_ms
    import torch
    t = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_bytes, steps, world, t_ms):
    """Whole-job GB/s: every rank decodes its own replica of the workload (no
    data-path exchange), so the job moves world * steps * step_bytes."""
    return step_bytes * steps * world / (t_ms / 1e3) / 1e9


def timed_span(stream, dev, n, body, flush):
    """Milliseconds of body(0) .. body(n - 1) enqueued on `stream`.  Without
    flush: one event pair around all of them.  With flush (inputs smaller
    than L2): each call gets its own event pair, and before each a write of
    twice L2 (outside the pairs) evicts what the previous call left in L2;
    the result is the sum of the pairs."""
    import torch
    if not flush:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            body(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    scratch = torch.empty((2 * l2 // 4 + 1024,), dtype=torch.int32, device=dev)
    pairs = []
    for i in range(n):
        scratch.fill_(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        body(i)
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs)


def l2_policy(dev, step_bytes):
    """(flush, description) for a decode step that reads step_bytes."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if step_bytes < l2:
        return True, ("L2 flushed before every timed step (a %.0f MB write outside the timed spans; the step reads "
                      "%.1f MB); each span is the step's device time, since the host issues the next step while "
                      "the flush runs" % (2 * l2 / 1e6, step_bytes / 1e6))
    return False, "inputs larger than L2 (%.0f MB per step)" % (step_bytes / 1e6)


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "decode_mma_traffic.json")


def recorded_traffic(step_bytes, workload, decode_impl):
    """DRAM bytes per scan launch from the committed ncu capture of this
    workload, scaled from the captured launch's algorithmic bytes to this
    run's mean step bytes; None when the kernel sources changed since the
    capture or no capture covers the run."""
    import hashlib
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
    except Exception:
        return None
    if h.hexdigest() != rec["sources_sha256"] or decode_impl == "simt":
        return None
    for r in rec["records"]:
        if r["applies_to"] == workload:
            return (r["dram_bytes_read"] + r["dram_bytes_write"]) / r["algorithmic_bytes"] * step_bytes
    return None


def _oracle_quant_rate(w, n_tok, threads):
    """bf16 K/V bytes in + page-block bytes out per second of the oracle's
    quantize-on-append (request 0's first n_tok tokens, every kv head), with
    `threads` independent oracle pools appending at once (one per thread)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from oracle.workload import kv_rows, request_bits
    H = w.num_kv_heads
    bits = request_bits(w, 0)[:n_tok]
    k, v = kv_rows(w, 0, 0, n_tok, list(range(H)))
    n2 = int((bits == 2).sum()) // 32 + 2
    n4 = -(-int((bits == 4).sum()) // 32) + n_tok // 32 + 4
    pools = [oracle.OraclePool(H, n2, n4, 1, n2 + n4) for _ in range(threads)]
    rids = [P.open() for P in pools]

    def one(i):
        assert pools[i].append(np.full(n_tok, rids[i]), bits, k, v) == oracle.OK

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:      # the oracle's calls release the GIL
        list(ex.map(one, range(threads)))
    dt = time.perf_counter() - t0
    ex0 = pools[0].export(rids[0], content=False)
    out_bytes = sum(3072 if is2 else 160 * int(f) for is2, f in zip(ex0["is_int2"], ex0["fill"])) * H
    in_bytes = n_tok * H * 128 * 2 * 2
    return (in_bytes + out_bytes) * threads / dt / 1e9, dt


def cpu_baseline(w, quant_tokens=8192):
    """The oracle as it stands, on this host's cores, over a bounded sample of
    the same workload, timed in two parts:
      quantize-on-append: request 0's first `quant_tokens` tokens (all kv
        heads) into a fresh oracle pool, one thread, then one pool per core
        appending at once (GB/s of bf16 K/V in + page blocks out);
      decode: fp64 attention of request 0 at its full context for the units
        (kv heads) of the sample, one thread over one unit, then all cores
        over two units with the oracle's OpenMP loop (KV-bytes GB/s, the
        metric's unit).
    value = the all-cores decode figure."""
    import oracle
    from oracle.workload import oracle_twin_for
    nproc = os.cpu_count() or 1
    q1, tq1 = _oracle_quant_rate(w, quant_tokens, 1)
    qn, tqn = _oracle_quant_rate(w, quant_tokens, nproc)
    heads = [0, 1] if w.num_kv_heads > 1 else [0]
    ow, pairs, nbytes = oracle_twin_for(w, heads=heads)
    q = ow.q(0)
    unit_pairs = pairs[:w.g]
    t0 = time.perf_counter()
    ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=unit_pairs, n_threads=1)
    td1 = time.perf_counter() - t0
    d1 = nbytes / len(heads) / td1 / 1e9
    cores = min(nproc, len(pairs))
    t0 = time.perf_counter()
    ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=pairs, n_threads=cores)
    tdn = time.perf_counter() - t0
    dn = nbytes / tdn / 1e9
    ctx = w.requests[0].n_prefill
    return {"value": dn, "unit": UNIT, "cores": cores, "kind": "oracle", "nproc": nproc,
            "sample": f"request 0 of {w.name}: quantize-on-append of its first {quant_tokens} tokens x "
                      f"{w.num_kv_heads} kv heads; fp64 decode of {len(heads)} kv-head unit(s) x {w.g} q heads "
                      f"at its full {ctx}-token context",
            "decode": {"single_thread_gbs": d1, "all_cores_gbs": dn, "threads": cores,
                       "single_thread_s": td1, "all_cores_s": tdn, "units": len(heads)},
            "quant": {"single_thread_gbs": q1, "all_cores_gbs": qn, "threads": nproc,
                      "single_thread_s": tq1, "all_cores_s": tqn, "tokens_per_pool": quant_tokens,
                      "unit": "GB/s of bf16 K/V in + page blocks out"}}


def run_reference(args):
    """Reference arm: the CPU oracle (the only reference this path has), as it
    stands, on this host's cores.  A step decodes one (request 0, kv head)
    unit at its full context: all g q heads on min(cores, g) OpenMP threads,
    or one q head when K such steps would take more than about two minutes."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import kvsynth
    from oracle.workload import oracle_twin_for
    w = kvsynth.make_workload(args.config)
    g = w.g
    ow, pairs, unit_bytes = oracle_twin_for(w, heads=[0])
    nproc = os.cpu_count() or 1
    cores = min(nproc, g)
    q = ow.q(0)
    t0 = time.perf_counter()
    ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=pairs, n_threads=cores)
    t_unit = time.perf_counter() - t0
    sample = pairs
    if args.steps * t_unit > 120.0:
        sample, cores = pairs[:1], 1
    step_bytes = unit_bytes * len(sample) / len(pairs)
    for _ in range(args.warmup):
        ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=sample, n_threads=cores)
    t0 = time.perf_counter()
    for s in range(args.steps):
        ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=sample, n_threads=cores)
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    desc = (f"one (request 0, kv head 0) unit of {w.name} per step at its full {w.requests[0].n_prefill}-token "
            f"context: {len(sample)} of its {g} q heads, fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                             "nproc": nproc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def context_desc(w):
    """Prefill context of the workload's requests: one length, or the range."""
    n = [r.n_prefill for r in w.requests]
    return n[0] if min(n) == max(n) else {"min": min(n), "max": max(n), "mean": float(np.mean(n))}


def budget_desc(w):
    """Average-bit budget B of the greedy allocator: one value, or the range over requests."""
    b = [num / den for num, den in (r.budget for r in w.requests)]
    return b[0] if min(b) == max(b) else {"min": min(b), "max": max(b), "mean": float(np.mean(b))}


def int2_fraction(gw):
    """Fraction of prefill tokens the allocator sent to INT2."""
    n2 = sum(int((b[:r.n_prefill] == 2).sum()) for b, r in zip(gw.bits, gw.w.requests))
    return n2 / max(1, sum(r.n_prefill for r in gw.w.requests))


def run_prefill(args):
    """Prefill of the workload's prompts in append calls of --chunk tokens (16K
    by default): of one request, or with --interleave one chunk of every
    request per call (chunk / requests tokens each, the shape of a batched
    chunked prefill).  Inputs resident in HBM: bf16 K and V rows read, page
    blocks written."""
    import torch
    import kvsynth
    from mixed_precision_kv_gb300.workload import GPUWorkload
    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    w = kvsynth.make_workload(args.config)
    H = w.num_kv_heads
    chunk = args.chunk
    times = []
    nreq = len(w.requests)
    per = max(32, chunk // nreq)   # --interleave: tokens of each request per call
    for rep_i in range(args.warmup + args.steps):
        gw = GPUWorkload(w, device=local, chunk=chunk)
        calls = []
        if args.interleave:
            for t0 in range(0, max(s.n_prefill for s in w.requests), per):
                ks, vs, rs, bs = [], [], [], []
                for r, spec in enumerate(w.requests):
                    n = min(per, spec.n_prefill - t0)
                    if n <= 0:
                        continue
                    k, v = gw.kv_rows(r, t0, n)
                    ks.append(k)
                    vs.append(v)
                    rs.append(np.full(n, gw.rids[r], np.int32))
                    bs.append(gw.bits[r][t0:t0 + n])
                calls.append((torch.cat(ks), torch.cat(vs), np.concatenate(rs), np.ascontiguousarray(np.concatenate(bs))))
        else:
            for r, spec in enumerate(w.requests):
                for t0 in range(0, spec.n_prefill, chunk):
                    n = min(chunk, spec.n_prefill - t0)
                    k, v = gw.kv_rows(r, t0, n)
                    calls.append((k, v, np.full(n, gw.rids[r], np.int32), np.ascontiguousarray(gw.bits[r][t0:t0 + n])))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k, v, rid, b in calls:
            gw.pool.append(k, v, rid, b)
        e1.record()
        torch.cuda.synchronize()
        if rep_i >= args.warmup:
            times.append(e0.elapsed_time(e1))
        n_tok = sum(s.n_prefill for s in w.requests)
        n_pages = sum(gw.pool.info(rid)[0] for rid in gw.rids)
        n2 = sum(int((gw.pool.export(rid, content=False)["is_int2"] == 1).sum()) for rid in gw.rids)
        del gw, calls
        torch.cuda.empty_cache()
    t_ms = float(np.median(times))
    in_bytes = n_tok * H * 128 * 2 * 2
    blk_bytes = (n2 * 3072 + (n_pages - n2) * 5120) * H
    peak, peak_kind = measured_peak()
    achieved = (in_bytes + blk_bytes) / (t_ms / 1e3) / 1e9
    line = {"metric": "prefill quantization: bf16 K/V bytes in + page blocks out, GB/s", "value": achieved,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, u4/u2 + f16 out",
            "data": "synthetic",
            "config": {"workload": w.name, "mode": "prefill", "tokens": n_tok, "num_kv_heads": H, "chunk": chunk,
                       "calls": ("one chunk of every request per call (%d tokens each)" % per if args.interleave
                                 else "one request per call"),
                       "tokens_per_s": n_tok / (t_ms / 1e3), "in_bytes": in_bytes, "out_bytes": blk_bytes},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                         "kernel": "whole prefill (append, direct INT2, repack, table scatter; host routing)"}}
    if rank == 0:
        print(json.dumps(line))
    return 0


def alloc_quality(w):
    """Synthetic distortion sum_k N_k D_k(b_k) of the prompts under the
    two-width and the three-width allocation at the same budget, and their
    average bits (the recipe's D tables stand in for a calibration)."""
    import mixed_precision_kv_gb300 as kvq
    from kvsynth.recipes import d3_table, tag_counts
    D3 = d3_table(w)
    D = np.stack([w.D2, D3, w.D4], 1)
    out = {"distortion_2w": 0.0, "distortion_3w": 0.0, "bits_2w": 0.0, "bits_3w": 0.0, "tokens": 0}
    for spec in w.requests:
        N = tag_counts(spec.tags[:spec.n_prefill])
        b2 = kvq.alloc_bits(N, w.D2, w.D4, spec.budget).astype(np.int64)
        b3 = kvq.alloc_bits3(N, w.D2, D3, w.D4, spec.budget).astype(np.int64)
        k = np.arange(N.size)
        out["distortion_2w"] += float((N * D[k, b2 - 2]).sum())
        out["distortion_3w"] += float((N * D[k, b3 - 2]).sum())
        out["bits_2w"] += float((N * b2).sum())
        out["bits_3w"] += float((N * b3).sum())
        out["tokens"] += int(N.sum())
    out["bits_2w"] /= out["tokens"]
    out["bits_3w"] /= out["tokens"]
    return out


def load_workload(args, total_steps):
    import kvsynth
    w = kvsynth.make_workload(args.config, steps=total_steps, n_req=args.requests or None)
    if args.requests:
        w.name = f"{w.name}-first{args.requests}"
    if args.q_heads:
        if args.q_heads % w.num_kv_heads or not 1 <= args.q_heads // w.num_kv_heads <= 8:
            raise SystemExit("--q-heads must be 1..8 times the workload's kv heads")
        w.name = f"{w.name}-q{args.q_heads}"
        w.num_q_heads = args.q_heads
    return w


def run_head_groups(args):
    """Head groups in pools of their own (Tangram: head groups keep different
    amounts of context).  The workload's kv heads are cut into N equal
    groups, one pool each, fed the group's rows of every token; group j keeps
    the most recent (j+1)/N of every prompt, evicts the older positions and
    drops its dead pages, so it holds only its own pages.  A step appends the
    new token to every pool, reorders, and decodes through one grouped call
    (one tensor-core scan over all pools).  The budgets are those of
    --ragged-heads when N = num_kv_heads, there held in one shared pool."""
    import torch
    import kvsynth
    import mixed_precision_kv_gb300 as kvq
    from mixed_precision_kv_gb300.workload import GroupWorkload

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    clk = ClockSampler(local).start()
    e2e_steps = max(args.steps // 4, 10)
    total_steps = args.warmup + args.steps + 3 + e2e_steps
    w = load_workload(args, total_steps)
    H, N = w.num_kv_heads, args.head_groups
    if N < 1 or N > 8 or H % N:
        raise SystemExit("--head-groups must divide the workload's kv heads, at most 8 groups")
    G = GroupWorkload(w, N, device=local, steps=total_steps)
    gw, pools, rids, hg, lo, keep = G.gw, G.pools, G.rids, G.hg, G.lo, G.keep
    B, Hq = len(w.requests), w.num_q_heads
    G.prefill()
    blocks_before = G.blocks()
    G.evict_and_drop()
    G.sync()
    blocks_after = G.blocks()
    dev = torch.device("cuda", local)
    kf = torch.empty((total_steps, B, H, 128), dtype=torch.bfloat16, device=dev)
    vf = torch.empty_like(kf)
    qs = torch.empty((total_steps, B, Hq, 128), dtype=torch.bfloat16, device=dev)
    bits = np.zeros((total_steps, B), np.uint8)
    for s in range(total_steps):
        for r in range(B):
            pos = w.requests[r].n_prefill + s
            kvsynth.fill_bf16_dev(kf[s, r].data_ptr(), 1, H, 128, w.seed, kvsynth.TENSOR_K, w.requests[r].stream,
                                  pos, gw.chan.data_ptr())
            kvsynth.fill_bf16_dev(vf[s, r].data_ptr(), 1, H, 128, w.seed, kvsynth.TENSOR_V, w.requests[r].stream,
                                  pos)
            bits[s, r] = gw.bits[r][pos]
        kvsynth.fill_bf16_dev(qs[s].data_ptr(), B, Hq, 128, w.seed, kvsynth.TENSOR_Q, s)
    ks = [kf[:, :, lo[j]:lo[j + 1]].contiguous() for j in range(N)]   # each group's rows, resident per step
    vs = [vf[:, :, lo[j]:lo[j + 1]].contiguous() for j in range(N)]
    del kf, vf
    rid_mat = np.stack(rids)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(s, kk=None, vv=None, q=None):
        for j, p in enumerate(pools):
            p.append(ks[j][s] if kk is None else kk[j], vs[j][s] if vv is None else vv[j], rids[j], bits[s])
            p.reorder(rids[j])
        return kvq.KVPool.decode_groups(pools, qs[s] if q is None else q, rid_mat, w.softmax_scale, out=out)

    def kv_bytes():
        return sum(p.last_decode_stats()["kv_bytes"] for p in pools)

    for s in range(args.warmup):
        step(s)
    for p in pools:
        p.sync()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s0 = args.warmup
    kv_first = kv_bytes()
    launches0 = sum(p.launch_count() for p in pools)
    timing_every = 1 if args.steps < 200 else 8
    pools[0].decode_timing(True, every=timing_every)
    flush, l2_desc = l2_policy(dev, kv_first)
    torch.cuda.synchronize()
    t_loop = timed_span(stream, dev, args.steps, lambda i: step(s0 + i), flush)
    clk.stop()
    if dist:
        dist.barrier()
    kv_last = kv_bytes()
    launches = sum(p.launch_count() for p in pools) - launches0
    n_timed, scan_ms, dec_ms = pools[0].decode_timing(False)
    for p in pools:
        p.sync()
    t_ms = reduce_max_time(t_loop, dist, dev)
    step_bytes = 0.5 * (kv_first + kv_last)
    value = job_throughput(step_bytes, args.steps, ws, t_ms)
    achieved = step_bytes / (scan_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()

    # end to end: one pinned host buffer per step (every group's K, then V, then q)
    s_e = s0 + args.steps + 3
    nk = B * hg * 128
    nq = qs[0].numel()
    parts = [x[s_e:s_e + e2e_steps].reshape(e2e_steps, nk) for x in ks + vs]
    hbuf = torch.cat(parts + [qs[s_e:s_e + e2e_steps].reshape(e2e_steps, nq)], dim=1).cpu().pin_memory()
    hout = torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory()
    dbuf = torch.empty((2 * N * nk + nq,), dtype=torch.bfloat16, device=dev)
    dk = [dbuf[j * nk:(j + 1) * nk].view(B, hg, 128) for j in range(N)]
    dv = [dbuf[(N + j) * nk:(N + j + 1) * nk].view(B, hg, 128) for j in range(N)]
    dq = dbuf[2 * N * nk:].view(qs[0].shape)
    for i in range(3):
        step(s0 + args.steps + i)
    torch.cuda.synchronize()
    e_first = kv_bytes()

    def e2e_step(i):
        dbuf.copy_(hbuf[i], non_blocking=True)
        step(s_e + i, dk, dv, dq)
        hout.copy_(out, non_blocking=True)

    e_ms = timed_span(stream, dev, e2e_steps, e2e_step, flush)
    e_last = kv_bytes()
    e_ms = reduce_max_time(e_ms, dist, dev)
    e2e_val = job_throughput(0.5 * (e_first + e_last), e2e_steps, ws, e_ms)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4/u2 codes, f16 meta, f32 accum", "data": "synthetic",
            "config": {"workload": f"{w.name}+head-groups{N}", "batch": B, "num_q_heads": Hq, "num_kv_heads": H,
                       "head_dim": 128, "context": context_desc(w), "page_tokens": 32, "budget_bits": budget_desc(w),
                       "decode_impl": "mma (grouped scan)",
                       "l2": l2_desc,
                       "us_per_layer_step": t_ms / args.steps * 1e3, "decode_us": dec_ms * 1e3,
                       "scan_us": scan_ms * 1e3, "decode_calls_timed": n_timed,
                       "pct_of_8000_gbs": value / ws / 8000 * 100},
            "head_groups": {"groups": N, "kv_heads_per_group": hg, "keep_fraction_of_prompt": keep,
                            "page_blocks_before_drop": blocks_before, "page_blocks_after_drop": blocks_after,
                            "kv_bytes_counted": "page blocks each group reads (its kept pages), table entries, "
                                                "q and out"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                         "kernel": "decode_mma_kernel (grouped split scan); CUDA events recorded by the library "
                                   "on the launch stream around %s launch of the timed region"
                                   % ("every" if timing_every == 1 else "every 8th")},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": dbuf.numel() * 2,
                    "d2h_bytes_per_step": hout.numel() * 4},
            "gpu_launches": launches,
            "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3,
                    help="workload 1..5 (default 3: batch 16, 64/8 heads, 100K tokens per request)")
    ap.add_argument("--requests", type=int, default=0,
                    help="run only the workload's first N requests (smaller cases for profiling)")
    ap.add_argument("--q-heads", type=int, default=0,
                    help="override the workload's number of query heads (GQA ratio = q heads / kv heads)")
    ap.add_argument("--decode-impl", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--segments", action="store_true",
                    help="decode with full-precision segments: per kv head 5%% vertical-line tokens excluded from "
                         "its quantized set, a 128-token window and a 128-token staging buffer in bf16; every "
                         "128 steps the staging buffer is quantized into the pool")
    ap.add_argument("--ragged-heads", action="store_true",
                    help="per-head budgets: kv head h keeps the most recent (h+1)/num_kv_heads of every prompt; "
                         "the older positions are excluded for that head only (whole pages are skipped)")
    ap.add_argument("--head-groups", type=int, default=0,
                    help="N > 0: the kv heads in N pools of their own; group j keeps the most recent (j+1)/N of "
                         "every prompt and drops its dead pages; one grouped decode per step")
    ap.add_argument("--int3-share", type=float, default=0.0,
                    help="make a seeded fraction of the INT4 tokens INT3 (three-width pool; prefill and steps)")
    ap.add_argument("--fp4-share", type=float, default=0.0,
                    help="make a seeded fraction of the INT4 tokens FP4 (E2M1) (prefill and steps)")
    ap.add_argument("--alloc3", action="store_true",
                    help="allocate INT2/INT3/INT4 with the three-width greedy over the same budget (D(3) from "
                         "the input recipe)")
    ap.add_argument("--interleave", action="store_true",
                    help="--mode prefill: every call carries one chunk of each request (--chunk tokens in all)")
    ap.add_argument("--chunk", type=int, default=16384,
                    help="--mode prefill: tokens per kv_append_quant call (one request per call)")
    ap.add_argument("--mode", default="decode", choices=["decode", "prefill"],
                    help="decode: the decode-step line (default); prefill: bulk quantization of the workload's "
                         "prompts through kv_append_quant")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "prefill":
        return run_prefill(args)
    if args.head_groups:
        return run_head_groups(args)

    import torch
    import kvsynth
    import mixed_precision_kv_gb300 as kvq
    from mixed_precision_kv_gb300.workload import GPUWorkload

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    # clocks are sampled from here (workload build and warm-up included) to the
    # end of the timed region, so that a short timed region still has samples
    clk = ClockSampler(local).start()
    e2e_steps = max(args.steps // 4, 10)
    total_steps = args.warmup + args.steps + 3 + e2e_steps
    SEG_W = SEG_WS = 128   # HyQuant window W and staging capacity W_s
    extra = SEG_W if args.segments else 0   # the frozen window is quantized again by the first flush
    w = load_workload(args, total_steps)
    if args.int3_share > 0:
        w.name = f"{w.name}+int3-{args.int3_share:g}"
    if args.fp4_share > 0:
        w.name = f"{w.name}+fp4-{args.fp4_share:g}"
    if args.alloc3:
        w.name = f"{w.name}+alloc3"
    gw = GPUWorkload(w, device=local, steps=total_steps, extra_tokens=extra, int3_share=args.int3_share,
                     fp4_share=args.fp4_share, three_widths=args.alloc3)
    gw.pool.set_decode_impl({"auto": 0, "simt": 1, "mma": 2}[args.decode_impl])
    gw.prefill()
    gw.evict()
    n_vl = []
    if args.ragged_heads:
        H = w.num_kv_heads
        for r, spec in enumerate(w.requests):
            n = spec.n_prefill
            cuts = [n - int(round(n * (h + 1) / H)) for h in range(H)]
            pos = np.concatenate([np.arange(c, dtype=np.int64) for c in cuts])
            heads = np.concatenate([np.full(c, h, np.int32) for h, c in enumerate(cuts)])
            gw.pool.evict_head(np.full(pos.size, gw.rids[r], np.int32), pos, heads)
    if args.segments:
        win_k, win_v, n_vl = gw.freeze_segments(rho=0.05, window=SEG_W, staging=SEG_WS)
    gw.reorder()
    gw.pool.sync()
    B, Hkv, Hq = len(gw.rids), w.num_kv_heads, w.num_q_heads
    dev = torch.device("cuda", local)
    # Per-step inputs, resident in HBM before timing.
    ks = torch.empty((total_steps, B, Hkv, 128), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    qs = torch.empty((total_steps, B, Hq, 128), dtype=torch.bfloat16, device=dev)
    bits = np.zeros((total_steps, B), np.uint8)
    for s in range(total_steps):
        for r in range(B):
            pos = w.requests[r].n_prefill + s
            kvsynth.fill_bf16_dev(ks[s, r].data_ptr(), 1, Hkv, 128, w.seed, kvsynth.TENSOR_K, w.requests[r].stream,
                                  pos, gw.chan.data_ptr())
            kvsynth.fill_bf16_dev(vs[s, r].data_ptr(), 1, Hkv, 128, w.seed, kvsynth.TENSOR_V, w.requests[r].stream,
                                  pos)
            bits[s, r] = gw.bits[r][pos]
        kvsynth.fill_bf16_dev(qs[s].data_ptr(), B, Hq, 128, w.seed, kvsynth.TENSOR_Q, s)
    rids = np.array(gw.rids, np.int32)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(s, k=None, v=None, q=None):
        gw.pool.append(ks[s] if k is None else k, vs[s] if v is None else v, rids, bits[s])
        gw.pool.reorder(rids)
        return gw.pool.decode(qs[s] if q is None else q, rids, w.softmax_scale, out=out)

    # Decode step with full-precision segments (HyQuant, Algorithm 3): the new
    # token joins the window; once window + staging hold W + W_s tokens, the
    # oldest W_s (the staging buffer) leave the lists and are quantized into
    # the pool.  The lists' non-vertical-line part is a queue of W_s-token
    # blocks: the frozen prefill window first, then blocks of step tokens.
    seg = {"fill": SEG_W, "blocks": [None], "cur": 0, "cur_len": 0, "fp_tok": 0}
    if args.segments:
        win_bits = np.stack([gw.bits[r][w.requests[r].n_prefill - SEG_W:w.requests[r].n_prefill] for r in range(B)], 1)
        rids_blk = np.tile(rids, SEG_WS)

    def seg_step(s, k=None, v=None, q=None):
        gw.pool.fp_append(rids, ks[s] if k is None else k, vs[s] if v is None else v)
        if seg["cur_len"] == 0:
            seg["cur"] = s
        seg["cur_len"] += 1
        if seg["cur_len"] == SEG_WS:
            seg["blocks"].append(seg["cur"])
            seg["cur_len"] = 0
        seg["fill"] += 1
        if seg["fill"] == SEG_W + SEG_WS:
            a = seg["blocks"].pop(0)
            kb, vb, bb = (win_k, win_v, win_bits) if a is None else (ks[a:a + SEG_WS], vs[a:a + SEG_WS],
                                                                    bits[a:a + SEG_WS])
            for r in range(B):
                gw.pool.fp_drop(rids[r], n_vl[r], SEG_WS)
            gw.pool.append(kb.reshape(SEG_WS * B, Hkv, 128), vb.reshape(SEG_WS * B, Hkv, 128), rids_blk,
                           np.ascontiguousarray(bb).reshape(-1))
            gw.pool.reorder(rids)
            seg["fill"] -= SEG_WS
        seg["fp_tok"] += sum(n_vl) + B * seg["fill"]
        return gw.pool.decode(qs[s] if q is None else q, rids, w.softmax_scale, out=out)

    if args.segments:
        step = seg_step

    for s in range(args.warmup):
        step(s)
    gw.pool.sync()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s0 = args.warmup
    # kv bytes per step: host accounting of the tables, read before and after
    # the timed steps (a step adds one token per request, so bytes grow
    # linearly and the mean of the two ends is the mean step)
    fp_row = Hkv * 128 * 2 * 2   # bf16 K and V of one list token, all kv heads
    kv_raw_first = gw.pool.last_decode_stats()["kv_bytes"]   # the last warm-up decode's algorithmic bytes
    kv_first = kv_raw_first - (sum(n_vl) + B * seg["fill"]) * fp_row * args.segments
    seg["fp_tok"] = 0
    launches0 = gw.pool.launch_count()
    # library-recorded events around the scan and merge of the timed decodes:
    # every call when the timed region is short, else every 8th (an event
    # between scan and merge stops the merge's launch from overlapping the
    # scan's drain, so the other calls run without one)
    timing_every = 1 if args.steps < 200 else 8
    gw.pool.decode_timing(True, every=timing_every)
    flush, l2_desc = l2_policy(dev, kv_raw_first)

    def timed_step(i):
        s = s0 + i
        if args.segments:
            seg_step(s)
        else:
            gw.pool.append(ks[s], vs[s], rids, bits[s])
            gw.pool.reorder(rids)
            gw.pool.decode(qs[s], rids, w.softmax_scale, out=out)

    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    t_loop = timed_span(stream, dev, args.steps, timed_step, flush)
    torch.cuda.nvtx.range_pop()
    clk.stop()
    if dist:
        dist.barrier()
    kv_last = gw.pool.last_decode_stats()["kv_bytes"] - (sum(n_vl) + B * seg["fill"]) * fp_row * args.segments
    fp_mean = seg["fp_tok"] / args.steps * fp_row if args.segments else 0.0
    launches = gw.pool.launch_count() - launches0
    n_timed, scan_ms, dec_ms = gw.pool.decode_timing(False)
    gw.pool.sync()
    t_ms = reduce_max_time(t_loop, dist, dev)
    step_bytes = 0.5 * (kv_first + kv_last) + fp_mean
    value = job_throughput(step_bytes, args.steps, ws, t_ms)
    achieved = step_bytes / (scan_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = None if (args.segments or args.ragged_heads) else recorded_traffic(step_bytes, w.name, args.decode_impl)

    # End to end: host (pinned) inputs copied in and the output copied out every
    # step.  A step's K, V and q sit in one pinned buffer and go in one copy.
    s_e = s0 + args.steps + 3
    nk, nq = ks[0].numel(), qs[0].numel()
    hbuf = torch.cat([ks[s_e:s_e + e2e_steps].reshape(e2e_steps, nk), vs[s_e:s_e + e2e_steps].reshape(e2e_steps, nk),
                      qs[s_e:s_e + e2e_steps].reshape(e2e_steps, nq)], dim=1).cpu().pin_memory()
    hout = torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory()
    dbuf = torch.empty((2 * nk + nq,), dtype=torch.bfloat16, device=dev)
    dk = dbuf[:nk].view(ks[0].shape)
    dv = dbuf[nk:2 * nk].view(vs[0].shape)
    dq = dbuf[2 * nk:].view(qs[0].shape)
    for i in range(3):
        step(s0 + args.steps + i)
    torch.cuda.synchronize()
    e_first = gw.pool.last_decode_stats()["kv_bytes"]

    def e2e_step(i):
        dbuf.copy_(hbuf[i], non_blocking=True)
        step(s_e + i, dk, dv, dq)
        hout.copy_(out, non_blocking=True)

    e_ms = timed_span(stream, dev, e2e_steps, e2e_step, flush)
    e_last = gw.pool.last_decode_stats()["kv_bytes"]
    e_ms = reduce_max_time(e_ms, dist, dev)
    e2e_val = job_throughput(0.5 * (e_first + e_last), e2e_steps, ws, e_ms)
    h2d = (dk.numel() + dv.numel() + dq.numel()) * 2
    d2h = hout.numel() * 4

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4/u2 codes, f16 meta, f32 accum", "data": "synthetic",
            "config": {"workload": w.name + ("+fp-segments" if args.segments else "") +
                                   ("+ragged-heads" if args.ragged_heads else ""), "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": 128,
                       "context": context_desc(w), "page_tokens": 32, "budget_bits": budget_desc(w),
                       "int2_token_fraction": int2_fraction(gw),
                       "decode_impl": args.decode_impl, "l2": l2_desc,
                       "us_per_layer_step": t_ms / args.steps * 1e3, "decode_us": dec_ms * 1e3,
                       "scan_us": scan_ms * 1e3, "decode_calls_timed": n_timed,
                       "kv_bytes_last_warmup_decode": kv_raw_first,
                       "pct_of_8000_gbs": value / ws / 8000 * 100},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "kernel": "decode_mma_kernel (split scan); CUDA events recorded by the library on "
                                   "the launch stream around %s launch of the timed region"
                                   % ("every" if timing_every == 1 else "every 8th")},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            **({"segments": {"vertical_lines": "5% of the non-window prefix per kv head (seeded synthetic score)",
                             "window": SEG_W, "staging": SEG_WS, "list_bytes_per_step": fp_mean,
                             "kernels": "fp_segment_kernel + decode_mma_kernel, one scan time"}}
               if args.segments else {}),
            "clocks": clk.summary()}
    if args.int3_share > 0:
        line["config"]["int3_token_fraction"] = float(np.mean(np.concatenate(gw.bits) == 3))
    if args.fp4_share > 0:
        line["config"]["fp4_token_fraction"] = float(np.mean(np.concatenate(gw.bits) == 0xF4))
    if args.alloc3:
        line["config"]["int3_token_fraction"] = float(np.mean(np.concatenate(gw.bits) == 3))
        line["config"]["allocation"] = alloc_quality(w)
    if rank == 0 and not args.no_cpu_baseline and args.int3_share <= 0 and args.fp4_share <= 0 and not args.alloc3:
        try:
            line["cpu_baseline"] = cpu_baseline(w)
        except Exception as e:  # reported, not fatal
            line["cpu_baseline"] = {"error": repr(e)}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
