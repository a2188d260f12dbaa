"""Benchmark: one decode step of the mixed INT2/INT4 paged-KV path.

A step = append one new token per request (INT4 quantize-on-append into the
tail page) + INT2-first reorder + split-KV fused-dequant decode attention with
log-sum-exp merge, over the Qwen3-8B-shaped single-layer workload (batch 8,
32 query / 8 KV heads, head_dim 128, 32K context per request, INT2:INT4 from
the greedy allocator at B = 3).  The metric is algorithmic KV bytes per step
(codes + binary16 scale/zero of every page block read, table entries, q, out)
divided by the step time.

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
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


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


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "decode_mma_traffic.json")


def recorded_traffic(step_bytes, workload, decode_impl):
    """DRAM bytes per scan launch from the committed ncu capture, scaled from the
    captured launch's algorithmic bytes to this run's mean step bytes; None when
    the kernel sources changed since the capture or the run differs from it."""
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
    if h.hexdigest() != rec["sources_sha256"] or rec["workload"] != workload or decode_impl == "simt":
        return None
    traffic = rec["dram_bytes_read"] + rec["dram_bytes_write"]
    return traffic / rec["algorithmic_bytes"] * step_bytes


def cpu_baseline(w, seconds=12.0):
    """The oracle as it stands, on this host's cores, over one request (all
    heads) of the same workload: KV-bytes GB/s of its decode."""
    import oracle
    from oracle.workload import oracle_twin_for
    ow, pairs, nbytes = oracle_twin_for(w)
    cores = min(os.cpu_count() or 1, len(pairs))
    q = ow.q(0)
    t0 = time.perf_counter()
    reps = 0
    while True:
        ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=pairs, n_threads=cores)
        reps += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": nbytes * reps / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"request 0 ({w.requests[0].n_prefill} tokens), all {w.num_q_heads} q heads, fp64 decode "
                      f"x{reps} in {dt:.1f}s"}


def run_reference(args):
    """Reference arm: the CPU oracle (the only reference this path has)."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import kvsynth
    from oracle.workload import oracle_twin_for
    w = kvsynth.make_workload(args.config)
    ow, pairs, nbytes_all = oracle_twin_for(w)
    g = w.g
    unit_bytes = nbytes_all / w.num_kv_heads          # one kv head of request 0 (+ q/out share)
    cores = 1
    q = ow.q(0)
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=pairs[:1], n_threads=1)
    t0 = time.perf_counter()
    for s in range(args.steps):
        p = pairs[rng.integers(0, len(pairs))][None]
        ow.P.decode(q[:1], [ow.rids[0]], w.softmax_scale, pairs=p, n_threads=1)
    dt = time.perf_counter() - t0
    value = unit_bytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": f"one (request 0, q head) pair per step, 1 of {g} heads "
                                                     f"sharing a kv head; {w.requests[0].n_prefill} tokens"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one q head of request 0 per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_prefill(args):
    """Prefill of the workload's prompts (16K-token append calls), inputs
    resident in HBM: bf16 K and V rows read, page blocks written."""
    import torch
    import kvsynth
    from mixed_precision_kv_gb300.workload import GPUWorkload
    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    w = kvsynth.make_workload(args.config)
    H = w.num_kv_heads
    chunk = 16384
    times = []
    for rep_i in range(args.warmup + args.steps):
        gw = GPUWorkload(w, device=local, chunk=chunk)
        calls = []
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
                       "tokens_per_s": n_tok / (t_ms / 1e3), "in_bytes": in_bytes, "out_bytes": blk_bytes},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                         "kernel": "whole prefill (append, direct INT2, repack, table scatter; host routing)"}}
    if rank == 0:
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--decode-impl", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--segments", action="store_true",
                    help="decode with full-precision segments: per kv head 5%% vertical-line tokens excluded from "
                         "its quantized set, a 128-token window and a 128-token staging buffer in bf16; every "
                         "128 steps the staging buffer is quantized into the pool")
    ap.add_argument("--ragged-heads", action="store_true",
                    help="per-head budgets: kv head h keeps the most recent (h+1)/num_kv_heads of every prompt; "
                         "the older positions are excluded for that head only (whole pages are skipped)")
    ap.add_argument("--mode", default="decode", choices=["decode", "prefill"],
                    help="decode: the decode-step line (default); prefill: bulk quantization of the workload's "
                         "prompts through kv_append_quant")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "prefill":
        return run_prefill(args)

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
    e2e_steps = max(args.steps // 4, 10)
    total_steps = args.warmup + args.steps + 3 + e2e_steps
    SEG_W = SEG_WS = 128   # HyQuant window W and staging capacity W_s
    extra = SEG_W if args.segments else 0   # the frozen window is quantized again by the first flush
    w = kvsynth.make_workload(args.config, steps=total_steps)
    gw = GPUWorkload(w, device=local, steps=total_steps, extra_tokens=extra)
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
    kv_first = gw.pool.last_decode_stats()["kv_bytes"] - (sum(n_vl) + B * seg["fill"]) * fp_row * args.segments
    seg["fp_tok"] = 0
    launches0 = gw.pool.launch_count()
    # library-recorded events around the scan and merge of every 8th timed
    # decode (an event between scan and merge stops the merge's launch from
    # overlapping the scan's drain, so the other calls run without one)
    gw.pool.decode_timing(True, every=8)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        start.record(stream)
        if args.segments:
            for i in range(args.steps):
                seg_step(s0 + i)
        else:
            for i in range(args.steps):
                s = s0 + i
                gw.pool.append(ks[s], vs[s], rids, bits[s])
                gw.pool.reorder(rids)
                gw.pool.decode(qs[s], rids, w.softmax_scale, out=out)
        end.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    if dist:
        dist.barrier()
    kv_last = gw.pool.last_decode_stats()["kv_bytes"] - (sum(n_vl) + B * seg["fill"]) * fp_row * args.segments
    fp_mean = seg["fp_tok"] / args.steps * fp_row if args.segments else 0.0
    launches = gw.pool.launch_count() - launches0
    n_timed, scan_ms, dec_ms = gw.pool.decode_timing(False)
    gw.pool.sync()
    t_ms = reduce_max_time(start.elapsed_time(end), dist, dev)
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
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        dbuf.copy_(hbuf[i], non_blocking=True)
        step(s_e + i, dk, dv, dq)
        hout.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e_last = gw.pool.last_decode_stats()["kv_bytes"]
    e_ms = reduce_max_time(e0.elapsed_time(e1), dist, dev)
    e2e_val = job_throughput(0.5 * (e_first + e_last), e2e_steps, ws, e_ms)
    h2d = (dk.numel() + dv.numel() + dq.numel()) * 2
    d2h = hout.numel() * 4

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4/u2 codes, f16 meta, f32 accum", "data": "synthetic",
            "config": {"workload": w.name + ("+fp-segments" if args.segments else "") +
                                   ("+ragged-heads" if args.ragged_heads else ""), "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": 128,
                       "context": w.requests[0].n_prefill, "page_tokens": 32, "budget_bits": "3.0",
                       "decode_impl": args.decode_impl, "l2": "inputs larger than L2 (%.0f MB per step)"
                                                             % (step_bytes / 1e6),
                       "us_per_layer_step": t_ms / args.steps * 1e3, "decode_us": dec_ms * 1e3,
                       "scan_us": scan_ms * 1e3, "decode_calls_timed": n_timed,
                       "pct_of_8000_gbs": value / ws / 8000 * 100},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "kernel": "decode_mma_kernel (split scan); CUDA events recorded by the library on "
                                   "the launch stream around every 8th launch of the timed region"},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            **({"segments": {"vertical_lines": "5% of the non-window prefix per kv head (seeded synthetic score)",
                             "window": SEG_W, "staging": SEG_WS, "list_bytes_per_step": fp_mean,
                             "kernels": "fp_segment_kernel + decode_mma_kernel, one scan time"}}
               if args.segments else {}),
            "clocks": clk.summary()}
    if rank == 0 and not args.no_cpu_baseline:
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
